"""GPU: the tensor-core router of large batches against the fp32 router and the oracle.

Both routers must give the same expert indices and the same gate-weight bits, and both must
match the oracle's routing exactly. The tensor-core router also reports, in the status words of
the workspace, how many tokens it had to recompute in full (a recomputed logit outside its
error bound) and the largest share of the bound any candidate logit used: the first must be 0
and the second well below 1 (the bound 2^-12 |x| |w| holds with room to spare)."""
import numpy as np
import pytest

import oracle
import routed_expert_ffn_moe_gb300 as moe
import synth
from gpu_helpers import TOL_TOPK_W, bf16_dev, to_dev, torch

pytestmark = pytest.mark.gpu

TC_ALWAYS, TC_NEVER = "1", "1000000000"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from routed_expert_ffn_moe_gb300 import build
    build.build()
    moe.load()


def route(monkeypatch, cfg, x, wg, bias, mode):
    monkeypatch.setenv("MOE_ROUTER_TC_MIN_TOKENS", mode)
    t = torch()
    s = moe.shape_of(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.n_shared, cfg.wdtype)
    ws = t.empty(moe.moe_workspace_size(s), dtype=t.uint8, device="cuda")
    idx = t.empty(cfg.T, cfg.k, dtype=t.int32, device="cuda")
    w = t.empty(cfg.T, cfg.k, dtype=t.float32, device="cuda")
    moe.moe_route(s, bf16_dev(x), bf16_dev(wg), to_dev(bias), idx, w, ws)
    moe.moe_check_device_status(ws)
    status = ws[:12].view(t.int32).cpu().numpy()
    return idx.cpu().numpy(), w.cpu().numpy(), status


def check_both(monkeypatch, cfg, x, wg, bias):
    i_tc, w_tc, st = route(monkeypatch, cfg, x, wg, bias, TC_ALWAYS)
    i_f, w_f, _ = route(monkeypatch, cfg, x, wg, bias, TC_NEVER)
    np.testing.assert_array_equal(i_tc, i_f)
    np.testing.assert_array_equal(w_tc.view(np.int32), w_f.view(np.int32))
    r_idx, _, r_w64 = oracle.route(oracle.router_logits(x, wg, bias), cfg.k)
    np.testing.assert_array_equal(i_tc, r_idx)
    np.testing.assert_allclose(w_tc, r_w64, rtol=0, atol=TOL_TOPK_W)
    full, use = int(st[1]), float(np.array([st[2]], np.int32).view(np.float32)[0])
    assert full == 0, f"{full} tokens recomputed in full"
    assert 0.0 <= use < 1.0 / 16, f"a candidate logit used {use:.3g} of its bound"
    return use


CASES = [
    {"T": 1024, "d": 7168, "E": 256, "k": 8},                       # the sweep's router
    {"T": 1000, "d": 7168, "E": 256, "k": 8, "router": "zipf"},    # ragged T, Zipf bias
    {"T": 300, "d": 7168, "E": 384, "k": 6},                        # V4-Pro's router width
    {"T": 70, "d": 1024, "E": 1024, "k": 32},                       # the widest E and k
    {"T": 65, "d": 16384, "E": 128, "k": 4},                        # the longest reduction
    {"T": 1, "d": 512, "E": 128, "k": 1},                           # one token, one choice
]


@pytest.mark.parametrize("over", CASES, ids=[str(c) for c in CASES])
def test_tc_router_equals_fp32_router_and_oracle(monkeypatch, over):
    cfg = synth.get_config("tiny", f=128, **over)
    use = check_both(monkeypatch, cfg, synth.host_x(cfg), synth.host_wg(cfg), synth.host_bias(cfg))
    print(f"largest share of the bound used: {use:.3g}")


def bf16_next(bits):
    """The next bf16 away from zero (one ulp), for finite nonzero values."""
    return (bits + 1).astype(np.uint16)


@pytest.mark.parametrize("bias", [False, True])
def test_tc_router_exact_and_near_ties_and_zero_tokens(monkeypatch, bias):
    # experts 128..255 repeat experts 0..127: every other pair exactly (equal logits, the lower
    # index must win), the rest one bf16 ulp apart in one element (logits a hair apart); tokens
    # 0..3 are zero rows (every logit equals the bias, or 0)
    cfg = synth.get_config("tiny", T=512, d=1024, E=256, k=8, f=128,
                           router="zipf" if bias else "uniform")
    x = synth.host_x(cfg).copy()
    x[:4] = 0
    wg = synth.host_wg(cfg).copy()
    wg[128:] = wg[:128]
    rng = np.random.default_rng(3)
    for e in range(129, 256, 2):
        i = int(rng.integers(cfg.d))
        if wg[e, i] & 0x7FFF:
            wg[e, i] = bf16_next(wg[e, i])
    check_both(monkeypatch, cfg, x, wg, synth.host_bias(cfg))


def test_tc_router_full_recomputation_path(monkeypatch):
    # A negative bound coefficient sends every token down the path a missed bound takes: all E
    # logits recomputed in the defined order. The counter says so, and the results are still
    # the fp32 router's bits.
    cfg = synth.get_config("tiny", T=1024, d=1024, E=256, k=8, f=128, router="zipf")
    x, wg, bias = synth.host_x(cfg), synth.host_wg(cfg), synth.host_bias(cfg)
    i_f, w_f, _ = route(monkeypatch, cfg, x, wg, bias, TC_NEVER)
    monkeypatch.setenv("MOE_ROUTER_TC_BOUND", "-1")
    i_tc, w_tc, st = route(monkeypatch, cfg, x, wg, bias, TC_ALWAYS)
    assert int(st[1]) == cfg.T
    np.testing.assert_array_equal(i_tc, i_f)
    np.testing.assert_array_equal(w_tc.view(np.int32), w_f.view(np.int32))
