"""Seeded synthetic inputs for the routed-expert MoE FFN layer.

The generator is a pure function of (seed, stream, element index), so any slice of any tensor
can be drawn on the host (for the CPU oracle) or on the GPU (for full-size workloads) with
bit-identical values. Stream ids: x = 1, router weight W_g = 2, expert gate/up weights w13 = 3,
expert down weights w2 = 4, Zipf popularity permutation = 6. The shared expert is expert index
E of w13 and w2, drawn from the same streams.

This module draws inputs only. It contains none of the layer's arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

from .configs import CONFIGS, MoeConfig, get_config, sweep_config  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.cu")
_LIB = os.path.join(_HERE, "libsynth.so")

STREAM_X, STREAM_WG, STREAM_W13, STREAM_W2, STREAM_ZIPF = 1, 2, 3, 4, 6
STREAM_HASH, STREAM_TOKEN_IDS = 7, 8
SIGMA_X, SIGMA_W = 1.0, 0.02


def build(force: bool = False) -> str:
    """Compile synth.cu (host + sm_103a device code) into libsynth.so next to it."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    cmd = ["nvcc", "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC,-fopenmp,-ffp-contract=off",
           "--fmad=false", "-gencode", "arch=compute_103a,code=sm_103a", _SRC, "-o", _LIB + ".tmp",
           "-lgomp"]
    subprocess.run(cmd, check=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        u64, i64, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        L.synth_key.restype = u64
        L.synth_key.argtypes = [u64, u64]
        L.synth_normal_bf16_host.restype = None
        L.synth_normal_bf16_host.argtypes = [vp, u64, u64, ctypes.c_double, u64]
        L.synth_normal_bf16_device.restype = ctypes.c_int
        L.synth_normal_bf16_device.argtypes = [vp, u64, u64, ctypes.c_double, u64, vp]
        L.synth_quant_e4m3_host.restype = None
        L.synth_quant_e4m3_host.argtypes = [vp, vp, vp, i64, i64]
        L.synth_quant_e4m3_device.restype = ctypes.c_int
        L.synth_quant_e4m3_device.argtypes = [vp, vp, vp, i64, i64, vp]
        L.synth_double_to_bf16_host.restype = None
        L.synth_double_to_bf16_host.argtypes = [vp, vp, i64]
        L.synth_f32_to_e4m3_host.restype = None
        L.synth_f32_to_e4m3_host.argtypes = [vp, vp, i64]
        L.synth_quant_mxfp4_host.restype = None
        L.synth_quant_mxfp4_host.argtypes = [vp, vp, vp, i64, i64]
        L.synth_quant_mxfp4_device.restype = ctypes.c_int
        L.synth_quant_mxfp4_device.argtypes = [vp, vp, vp, i64, i64, vp]
        L.synth_f32_to_e2m1_host.restype = None
        L.synth_f32_to_e2m1_host.argtypes = [vp, vp, i64]
        _lib = L
    return _lib


def key(seed: int, stream: int) -> int:
    return int(lib().synth_key(seed, stream))


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def normal_bf16(seed: int, stream: int, sigma: float, offset: int, n: int) -> np.ndarray:
    """Elements [offset, offset+n) of a stream, as bf16 bit patterns (uint16), on the host."""
    out = np.empty(n, dtype=np.uint16)
    if n:
        lib().synth_normal_bf16_host(_ptr(out), n, key(seed, stream), float(sigma), offset)
    return out


def double_to_bf16(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().synth_double_to_bf16_host(_ptr(v), _ptr(out), v.size)
    return out


def f32_to_e4m3(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().synth_f32_to_e4m3_host(_ptr(v), _ptr(out), v.size)
    return out


def quantize_e4m3(w_bf16: np.ndarray):
    """Block-quantise a row-major [rows, cols] bf16 matrix (uint16 bits) to E4M3 codes plus
    fp32 scales of shape [rows/128, cols/128]."""
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    rows, cols = w.shape
    assert rows % 128 == 0 and cols % 128 == 0
    q = np.empty((rows, cols), dtype=np.uint8)
    s = np.empty((rows // 128, cols // 128), dtype=np.float32)
    lib().synth_quant_e4m3_host(_ptr(w), _ptr(q), _ptr(s), rows, cols)
    return q, s


def f32_to_e2m1(v: np.ndarray) -> np.ndarray:
    """fp32 values -> E2M1 codes (one per uint8), round to nearest even, saturating to +-6."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().synth_f32_to_e2m1_host(_ptr(v), _ptr(out), v.size)
    return out


def quantize_mxfp4(w_bf16: np.ndarray):
    """MXFP4-quantise a row-major [rows, cols] bf16 matrix (uint16 bits): E2M1 code pairs
    [rows, cols/2] (element 2j in the low nibble) and E8M0 scales [rows, cols/32], one per 32
    consecutive elements of a row."""
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    rows, cols = w.shape
    assert cols % 32 == 0
    q = np.empty((rows, cols // 2), dtype=np.uint8)
    s = np.empty((rows, cols // 32), dtype=np.uint8)
    lib().synth_quant_mxfp4_host(_ptr(w), _ptr(q), _ptr(s), rows, cols)
    return q, s


def zipf_bias(E: int, seed: int, s: float = 1.1, alpha: float = 1.5) -> np.ndarray:
    """Per-expert router bias b[e] = alpha * ln(z_e), z_e proportional to rank_e^-s, where the
    ranks are a seeded Fisher-Yates permutation of the experts (SplitMix64 stream 6)."""
    k6 = key(seed, STREAM_ZIPF)
    perm = list(range(E))
    for i in range(E - 1, 0, -1):
        u = _splitmix_draw(k6, E - 1 - i)
        j = u % (i + 1)
        perm[i], perm[j] = perm[j], perm[i]
    rank = np.empty(E, dtype=np.float64)
    for r, e in enumerate(perm):
        rank[e] = r + 1
    z = rank ** (-s)
    z /= z.sum()
    return (alpha * np.log(z)).astype(np.float32)


def hash_table(vocab: int, E: int, k: int, seed: int = 0) -> np.ndarray:
    """A hash-routing table tid2eid [vocab, k] int32: row v holds k distinct experts, the first
    k of a Fisher-Yates shuffle of range(E) driven by SplitMix64 stream 7 (draws E*v onwards)."""
    kh = key(seed, STREAM_HASH)
    out = np.empty((vocab, k), dtype=np.int32)
    for v in range(vocab):
        perm = list(range(E))
        for i in range(k):
            j = i + _splitmix_draw(kh, E * v + i) % (E - i)
            perm[i], perm[j] = perm[j], perm[i]
        out[v] = perm[:k]
    return out


def token_ids(T: int, vocab: int, seed: int = 0) -> np.ndarray:
    """Token ids [T] int32 uniform in [0, vocab) (SplitMix64 stream 8)."""
    kt = key(seed, STREAM_TOKEN_IDS)
    return np.array([_splitmix_draw(kt, t) % vocab for t in range(T)], dtype=np.int32)


def _splitmix_draw(k: int, n: int) -> int:
    M = (1 << 64) - 1
    z = (k + (n + 1) * 0x9E3779B97F4A7C15) & M
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M
    return z ^ (z >> 31)


# ---------------------------------------------------------------------------------------------
# Host-side tensors for one config (small configs, or slices of big ones for the oracle).
# ---------------------------------------------------------------------------------------------

def host_x(cfg: MoeConfig, tokens=None) -> np.ndarray:
    """x [T, d] bf16 bits; `tokens` selects rows."""
    if tokens is None:
        return normal_bf16(cfg.seed, STREAM_X, SIGMA_X, 0, cfg.T * cfg.d).reshape(cfg.T, cfg.d)
    rows = [normal_bf16(cfg.seed, STREAM_X, SIGMA_X, int(t) * cfg.d, cfg.d) for t in tokens]
    return np.stack(rows) if rows else np.zeros((0, cfg.d), np.uint16)


def host_wg(cfg: MoeConfig) -> np.ndarray:
    return normal_bf16(cfg.seed, STREAM_WG, SIGMA_W, 0, cfg.E * cfg.d).reshape(cfg.E, cfg.d)


def host_bias(cfg: MoeConfig):
    return zipf_bias(cfg.E, cfg.seed) if cfg.router == "zipf" else None


def host_w13_expert(cfg: MoeConfig, e: int) -> np.ndarray:
    """Expert e's [2f, d] gate (rows 0..f-1) and up (rows f..2f-1) weights, bf16 bits."""
    n = 2 * cfg.f * cfg.d
    return normal_bf16(cfg.seed, STREAM_W13, SIGMA_W, e * n, n).reshape(2 * cfg.f, cfg.d)


def host_w2_expert(cfg: MoeConfig, e: int) -> np.ndarray:
    """Expert e's [d, f] down weights, bf16 bits."""
    n = cfg.d * cfg.f
    return normal_bf16(cfg.seed, STREAM_W2, SIGMA_W, e * n, n).reshape(cfg.d, cfg.f)


@dataclass
class ExpertWeights:
    """One expert's weights as stored on the device: bf16 bits, E4M3 codes + fp32 scales, or
    E2M1 code pairs + E8M0 scales."""
    w13: np.ndarray
    w2: np.ndarray
    s13: np.ndarray | None = None
    s2: np.ndarray | None = None


def host_expert(cfg: MoeConfig, e: int) -> ExpertWeights:
    w13, w2 = host_w13_expert(cfg, e), host_w2_expert(cfg, e)
    if cfg.wdtype == "bf16":
        return ExpertWeights(w13, w2)
    if cfg.wdtype == "mxfp4":
        q13, s13 = quantize_mxfp4(w13)
        q2, s2 = quantize_mxfp4(w2)
        return ExpertWeights(q13, q2, s13, s2)
    q13, s13 = quantize_e4m3(w13)
    q2, s2 = quantize_e4m3(w2)
    return ExpertWeights(q13, q2, s13, s2)


@dataclass
class HostInputs:
    x: np.ndarray
    wg: np.ndarray
    bias: np.ndarray | None
    experts: list = field(default_factory=list)


def host_inputs(cfg: MoeConfig) -> HostInputs:
    """All inputs of a (small) config on the host."""
    n_exp = cfg.E + cfg.n_shared
    return HostInputs(host_x(cfg), host_wg(cfg), host_bias(cfg),
                      [host_expert(cfg, e) for e in range(n_exp)])


# ---------------------------------------------------------------------------------------------
# Device-side tensors (torch) for full-size workloads.
# ---------------------------------------------------------------------------------------------

def _dev_normal(t, seed, stream, sigma, offset=0):
    import torch
    rc = lib().synth_normal_bf16_device(t.data_ptr(), t.numel(), key(seed, stream), float(sigma),
                                        offset, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if rc:
        raise RuntimeError(f"synth device generator failed: cuda error {rc}")
    return t


def device_inputs(cfg: MoeConfig, device="cuda"):
    """Draw every input of a config directly into HBM. Returns a dict of torch tensors:
    x [T,d] bf16, wg [E,d] bf16, bias [E] f32 or None, w13 [E+S,2f,d], w2 [E+S,d,f] (bf16, or
    uint8 E4M3 codes), s13 [E+S,2f/128,d/128], s2 [E+S,d/128,f/128] f32 or None; for MXFP4,
    w13 [E+S,2f,d/2] and w2 [E+S,d,f/2] uint8 code pairs with s13 [E+S,2f,d/32] and
    s2 [E+S,d,f/32] uint8 E8M0 scales."""
    import torch
    n_exp = cfg.E + cfg.n_shared
    x = _dev_normal(torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device=device),
                    cfg.seed, STREAM_X, SIGMA_X)
    wg = _dev_normal(torch.empty(cfg.E, cfg.d, dtype=torch.bfloat16, device=device),
                     cfg.seed, STREAM_WG, SIGMA_W)
    b = host_bias(cfg)
    bias = torch.from_numpy(b).to(device) if b is not None else None
    out = {"x": x, "wg": wg, "bias": bias}
    for name, stream, shape in (("w13", STREAM_W13, (n_exp, 2 * cfg.f, cfg.d)),
                                ("w2", STREAM_W2, (n_exp, cfg.d, cfg.f))):
        if cfg.wdtype == "bf16":
            out[name] = _dev_normal(torch.empty(*shape, dtype=torch.bfloat16, device=device),
                                    cfg.seed, stream, SIGMA_W)
            out["s" + name[1:]] = None
            continue
        fp4 = cfg.wdtype == "mxfp4"
        if fp4:
            q = torch.empty(shape[0], shape[1], shape[2] // 2, dtype=torch.uint8, device=device)
            s = torch.empty(shape[0], shape[1], shape[2] // 32, dtype=torch.uint8, device=device)
        else:
            q = torch.empty(*shape, dtype=torch.uint8, device=device)
            s = torch.empty(shape[0], shape[1] // 128, shape[2] // 128, dtype=torch.float32,
                            device=device)
        quant = lib().synth_quant_mxfp4_device if fp4 else lib().synth_quant_e4m3_device
        # quantise one expert at a time so the bf16 staging buffer stays small
        stage = torch.empty(shape[1], shape[2], dtype=torch.bfloat16, device=device)
        per = shape[1] * shape[2]
        cs = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        for e in range(n_exp):
            _dev_normal(stage, cfg.seed, stream, SIGMA_W, offset=e * per)
            rc = quant(stage.data_ptr(), q[e].data_ptr(), s[e].data_ptr(), shape[1], shape[2], cs)
            if rc:
                raise RuntimeError(f"synth device quantiser failed: cuda error {rc}")
        del stage
        out[name] = q
        out["s" + name[1:]] = s
    return out


__all__ = ["CONFIGS", "MoeConfig", "get_config", "sweep_config", "build", "normal_bf16",
           "quantize_e4m3", "quantize_mxfp4", "f32_to_e2m1", "zipf_bias", "hash_table",
           "token_ids", "host_inputs", "host_expert", "host_x", "host_wg",
           "host_bias", "device_inputs", "ExpertWeights", "HostInputs"]
