"""Shared helpers of the GPU tests: move seeded inputs to the device, run the layer through the C
ABI one call at a time, and compare with the oracle."""
from __future__ import annotations

import numpy as np

import oracle
import synth

# Acceptance bars of the layer output y (bf16) against the fp64 oracle.
TOL_MAX_ABS_BF16 = 2e-2
TOL_REL_L2_BF16 = 1e-2
TOL_REL_L2_FP8 = 3e-2
# MXFP4 weights enter the products exactly and the activations carry about one bf16 rounding
# (two E4M3 terms per element), so the bf16 bars apply to them too.
# gate weights: fp32 softmax over the k chosen logits vs the fp64 renormalised softmax
TOL_TOPK_W = 2e-6


def torch():
    import torch as _t
    return _t


def bf16_dev(a: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a).view(np.int16)).to("cuda").view(t.bfloat16)


def bf16_host(t) -> np.ndarray:
    return t.detach().view(torch().int16).cpu().numpy().view(np.uint16)


def to_dev(a):
    return None if a is None else torch().from_numpy(np.ascontiguousarray(a)).to("cuda")


def device_weights(cfg, inp: synth.HostInputs) -> dict:
    """Stacked [E+S, ...] device weights from host-drawn per-expert weights (small configs)."""
    w13 = np.ascontiguousarray(np.stack([e.w13 for e in inp.experts]))
    w2 = np.ascontiguousarray(np.stack([e.w2 for e in inp.experts]))
    out = {"wg": bf16_dev(inp.wg), "bias": to_dev(inp.bias)}
    if cfg.wdtype == "bf16":
        out.update(w13=bf16_dev(w13), w2=bf16_dev(w2), s13=None, s2=None)
    else:
        out.update(w13=to_dev(w13), w2=to_dev(w2),
                   s13=to_dev(np.stack([e.s13 for e in inp.experts])),
                   s2=to_dev(np.stack([e.s2 for e in inp.experts])))
    return out


def rel_l2(a, b) -> float:
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a - b))


def bf16_half_ulp(v):
    """Half the spacing of bf16 numbers at |v|: the largest error of rounding v to bf16."""
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 8)


def assert_y_close(y_gpu_bits, y_ref, wdtype, what="y"):
    """The layer output is bf16, so each element carries the format's own rounding on top of
    the computation error: the max-abs bar is 2e-2 for the computation plus that half-ulp
    (|y| reaches ~10 at the V3 shapes, where a bf16 half-ulp is 0.031)."""
    y = oracle.bf16_to_f64(y_gpu_bits)
    if not y.size:
        return 0.0, 0.0
    err = np.abs(y - y_ref)
    ma = float(err.max())
    excess = float((err - bf16_half_ulp(y_ref)).max())
    rl = rel_l2(y, y_ref)
    if wdtype in ("bf16", "mxfp4"):
        assert excess <= TOL_MAX_ABS_BF16 and rl <= TOL_REL_L2_BF16, (what, ma, excess, rl)
    else:
        assert rl <= TOL_REL_L2_FP8, (what, ma, rl)
    return ma, rl
