"""GPU parity: each C-ABI call and the whole layer against the CPU oracle, on seeded inputs.

Routing indices and the permutation must match bit for bit; gate weights within 2e-6; the
layer output within max-abs 2e-2 and relative-L2 1e-2 (bf16 and MXFP4 weights) or relative-L2
3e-2 (FP8 weights) of the fp64 oracle."""
import numpy as np
import pytest

import oracle
import routed_expert_ffn_moe_gb300 as moe
import synth
from gpu_helpers import (TOL_TOPK_W, assert_y_close, bf16_dev, bf16_host, device_weights,
                         rel_l2, to_dev, torch)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from routed_expert_ffn_moe_gb300 import build
    build.build()
    moe.load()


def run_layer(cfg, x_dev, w):
    """The four calls in order; returns the MoeLayer with every intermediate on the device."""
    layer = moe.MoeLayer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.n_shared, cfg.wdtype, w)
    layer.forward(x_dev)
    torch().cuda.synchronize()
    moe.moe_check_device_status(layer.ws)
    return layer


def check_small(cfg, bias_override=None):
    inp = synth.host_inputs(cfg)
    if bias_override is not None:
        inp.bias = bias_override
    ref = oracle.moe_layer(cfg, inp)
    w = device_weights(cfg, inp)
    layer = run_layer(cfg, bf16_dev(inp.x), w)
    T, k = cfg.T, cfg.k
    idx = layer.topk_idx.cpu().numpy()
    np.testing.assert_array_equal(idx, ref["topk_idx"])
    np.testing.assert_allclose(layer.topk_w.cpu().numpy(), ref["topk_w64"], rtol=0, atol=TOL_TOPK_W)
    np.testing.assert_array_equal(layer.expert_offsets.cpu().numpy(), ref["expert_offsets"])
    np.testing.assert_array_equal(layer.perm_token.cpu().numpy()[: T * k], ref["perm_token"])
    np.testing.assert_array_equal(layer.inv_slot.cpu().numpy()[: T * k], ref["inv_slot"])
    yp = layer.y_perm.cpu().numpy()[: cfg.slots]
    if cfg.slots:
        assert rel_l2(yp, ref["y_perm"]) <= 1e-2
    assert_y_close(bf16_host(layer.y), ref["y"], cfg.wdtype)
    return layer, ref


SMALL = [
    ("tiny", {}),
    ("tiny", {"wdtype": "fp8"}),
    ("tiny", {"router": "zipf", "T": 45}),
    ("tiny", {"n_shared": 0}),
    ("tiny", {"k": 8}),                        # k = E: every expert
    ("tiny", {"E": 1, "k": 1}),                # a single expert
    ("tiny", {"T": 1}),
    ("tiny", {"T": 37}),                       # ragged: not a multiple of 32 or 4
    ("tiny", {"T": 0}),
    ("tiny", {"d": 512, "f": 384, "T": 70, "E": 12, "k": 3}),
    ("tiny", {"d": 512, "f": 384, "T": 70, "E": 12, "k": 3, "wdtype": "fp8"}),
    ("tiny", {"T": 100, "E": 8, "k": 2, "wdtype": "fp8"}),   # 64-token FP8 decode tiles
    ("tiny", {"T": 40, "d": 384, "f": 256, "E": 8, "k": 2, "wdtype": "fp8"}),  # single down tiles
    ("tiny", {"T": 300, "E": 40, "k": 5}),     # several permute chunks, uneven segments
    # FP8 prefill tiles (more than 32 routed slots per expert): paired and single down tiles
    ("tiny", {"T": 600, "E": 8, "k": 2, "wdtype": "fp8"}),
    # FP8 prefill tiles on CTA pairs (even m-tile counts in both passes), full and ragged token
    # tiles; MXFP4 prefill on CTA pairs
    ("tiny", {"T": 600, "d": 512, "f": 256, "E": 8, "k": 2, "wdtype": "fp8"}),
    ("tiny", {"T": 600, "d": 1024, "f": 512, "E": 8, "k": 2, "wdtype": "fp8"}),
    ("tiny", {"T": 1500, "d": 512, "f": 256, "E": 8, "k": 2, "wdtype": "fp8", "router": "zipf"}),
    ("tiny", {"T": 600, "d": 512, "f": 256, "E": 8, "k": 2, "wdtype": "mxfp4"}),
    ("tiny", {"T": 600, "d": 512, "f": 256, "E": 8, "k": 2}),                  # bf16 pairs
    # bf16 prefill split: cold experts on decode tiles beside hot ones on paired tiles
    ("tiny", {"router": "zipf", "T": 600, "d": 512, "f": 256, "E": 16, "k": 2}),
    ("tiny", {"T": 333, "d": 384, "f": 256, "E": 6, "k": 3, "wdtype": "fp8"}),
    ("tiny", {"T": 333, "d": 384, "f": 256, "E": 6, "k": 3}),
    # MXFP4 weights: block-scaled MMAs on 16-, 32- and 48-token decode tiles (paired and single
    # down tiles, one or two K slices per stage), f16 prefill tiles, ragged and degenerate batches
    ("tiny", {"wdtype": "mxfp4"}),
    ("tiny", {"T": 10, "d": 384, "f": 256, "E": 8, "k": 2, "wdtype": "mxfp4"}),
    ("tiny", {"T": 100, "d": 384, "f": 256, "E": 8, "k": 2, "wdtype": "mxfp4"}),
    ("tiny", {"T": 40, "d": 384, "f": 256, "E": 8, "k": 2, "wdtype": "mxfp4"}),
    ("tiny", {"d": 512, "f": 384, "T": 70, "E": 12, "k": 3, "wdtype": "mxfp4"}),
    ("tiny", {"T": 600, "E": 8, "k": 2, "wdtype": "mxfp4"}),
    ("tiny", {"T": 333, "d": 384, "f": 256, "E": 6, "k": 3, "wdtype": "mxfp4"}),
    ("tiny", {"router": "zipf", "T": 45, "wdtype": "mxfp4"}),
    ("tiny", {"T": 1, "wdtype": "mxfp4"}),
    ("tiny", {"T": 0, "wdtype": "mxfp4"}),
    ("tiny", {"n_shared": 0, "T": 37, "wdtype": "mxfp4"}),
    # a batch large enough for the tensor-core router (E a multiple of 128), with the shared
    # expert's FFN overlapping it on the second stream
    ("tiny", {"T": 1100, "d": 512, "f": 256, "E": 128, "k": 4}),
    ("tiny", {"T": 1100, "d": 512, "f": 256, "E": 128, "k": 4, "router": "zipf", "wdtype": "fp8"}),
]


@pytest.mark.parametrize("name,over", SMALL, ids=[str(o) for _, o in SMALL])
def test_small_layer_matches_oracle(name, over):
    check_small(synth.get_config(name, **over))


@pytest.mark.parametrize("tc_min", ["3", "1000000000"])
@pytest.mark.parametrize("over", [{}, {"wdtype": "fp8"}, {"T": 70, "d": 512, "f": 384, "E": 12, "k": 3},
                                  {"T": 70, "d": 512, "f": 384, "E": 12, "k": 3, "wdtype": "fp8"}],
                         ids=["bf16", "fp8", "bf16_big", "fp8_big"])
def test_weight_streaming_path_and_mixed_split(monkeypatch, tc_min, over):
    # experts below tc_min tokens run on the weight-streaming GEMV, the rest on tensor cores
    monkeypatch.setenv("MOE_TC_MIN_TOKENS", tc_min)
    check_small(synth.get_config("tiny", **over))


def test_all_tokens_to_one_expert():
    cfg = synth.get_config("tiny", T=40, k=1, router="zipf")
    bias = np.zeros(cfg.E, np.float32)
    bias[5] = 100.0
    layer, ref = check_small(cfg, bias_override=bias)
    off = layer.expert_offsets.cpu().numpy()
    assert off[6] - off[5] == 40 and off[5] == 0


def test_permute_direct_random_rows():
    rng = np.random.default_rng(11)
    for T, E, k, S in ((1, 1, 1, 1), (33, 7, 7, 0), (257, 64, 6, 1), (1000, 384, 6, 1)):
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        s = moe.shape_of(T, 256, E, k, 128, S)
        ws = torch().empty(moe.moe_workspace_size(s), dtype=torch().uint8, device="cuda")
        ws[:4].zero_()
        off = torch().empty(E + 2, dtype=torch().int32, device="cuda")
        perm = torch().empty(T * k, dtype=torch().int32, device="cuda")
        inv = torch().empty(T * k, dtype=torch().int32, device="cuda")
        moe.moe_permute(s, to_dev(idx), off, perm, inv, ws)
        torch().cuda.synchronize()
        moe.moe_check_device_status(ws)
        r_off, r_perm, r_inv = oracle.permute(idx, E, S)
        np.testing.assert_array_equal(off.cpu().numpy(), r_off)
        np.testing.assert_array_equal(perm.cpu().numpy(), r_perm)
        np.testing.assert_array_equal(inv.cpu().numpy(), r_inv)


def test_permute_flags_out_of_range_expert_without_faulting():
    T, E, k = 8, 4, 2
    idx = np.tile(np.array([[0, 1]], np.int32), (T, 1))
    idx[3, 1] = E          # out of range
    idx[5, 1] = 0          # repeats the row's first choice
    s = moe.shape_of(T, 256, E, k, 128, 1)
    ws = torch().zeros(moe.moe_workspace_size(s), dtype=torch().uint8, device="cuda")
    off = torch().empty(E + 2, dtype=torch().int32, device="cuda")
    perm = torch().zeros(T * k, dtype=torch().int32, device="cuda")
    inv = torch().empty(T * k, dtype=torch().int32, device="cuda")
    moe.moe_permute(s, to_dev(idx), off, perm, inv, ws)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_check_device_status(ws)
    assert ei.value.status == -6
    inv_h = inv.cpu().numpy().reshape(T, k)
    assert inv_h[3, 1] == -1 and inv_h[5, 1] == -1
    moe.moe_check_device_status(ws)  # the check cleared the flag


def test_bounded_wait_gives_up_and_reports_timeout():
    # A device wait that nothing completes must give up after its limit, record the timeout in
    # the status word and leave the context usable (no trap, no hang).
    import time
    s = moe.shape_of(16, 256, 8, 2, 128, 1)
    ws = torch().zeros(moe.moe_workspace_size(s), dtype=torch().uint8, device="cuda")
    t0 = time.perf_counter()
    moe.moe_selftest_bounded_wait(ws, 50_000)
    torch().cuda.synchronize()
    waited = time.perf_counter() - t0
    assert 0.04 <= waited < 5.0
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_check_device_status(ws)
    assert ei.value.status == -5
    moe.moe_check_device_status(ws)  # the check cleared the word
    # the context still runs the layer correctly afterwards
    check_small(synth.get_config("tiny"))


def test_combine_direct():
    rng = np.random.default_rng(12)
    T, k, d, S = 50, 4, 384, 1
    idx = np.stack([rng.permutation(16)[:k] for _ in range(T)]).astype(np.int32)
    _, _, inv = oracle.permute(idx, 16, S)
    yp = rng.normal(size=(T * k + S * T, d)).astype(np.float32)
    w = rng.dirichlet(np.ones(k), size=T).astype(np.float32)
    s = moe.shape_of(T, d, 16, k, 128, S)
    ws = torch().zeros(moe.moe_workspace_size(s), dtype=torch().uint8, device="cuda")
    y = torch().empty(T, d, dtype=torch().bfloat16, device="cuda")
    moe.moe_combine(s, to_dev(yp), to_dev(inv), to_dev(w), y, ws)
    torch().cuda.synchronize()
    ref = oracle.combine(yp.astype(np.float64), inv, w.astype(np.float64), T, k, S)
    got = oracle.bf16_to_f64(bf16_host(y))
    # one bf16 rounding of the fp32 sum: |err| <= 2^-8 |y| + fp32 accumulation error
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-5)


@pytest.mark.parametrize("over", [{}, {"wdtype": "fp8"},
                                  # decode batches of at most 8 tokens: the fused front
                                  {"T": 1, "wdtype": "fp8"}, {"T": 8, "E": 40, "k": 6},
                                  {"T": 7, "E": 384, "k": 6, "wdtype": "mxfp4"},
                                  {"T": 8, "E": 1024, "k": 32, "d": 256, "f": 128},
                                  {"T": 32, "E": 40, "k": 6},
                                  {"router": "zipf", "T": 600, "d": 512, "f": 256, "E": 16, "k": 2},
                                  {"T": 600, "d": 512, "f": 256, "E": 8, "k": 2, "wdtype": "fp8"},
                                  {"n_shared": 0}, {"wdtype": "mxfp4"},
                                  {"T": 600, "d": 512, "f": 256, "E": 8, "k": 2, "wdtype": "mxfp4"},
                                  {"T": 1100, "d": 512, "f": 256, "E": 128, "k": 4}])
def test_forward_equals_the_four_calls(over):
    # moe_forward runs the shared expert on its own stream: every output must be bit-identical
    # to the four separate calls.
    cfg = synth.get_config("tiny", **over)
    inp = synth.host_inputs(cfg)
    w = device_weights(cfg, inp)
    x = bf16_dev(inp.x)
    one = moe.MoeLayer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.n_shared, cfg.wdtype, w)
    four = moe.MoeLayer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.n_shared, cfg.wdtype, w)
    one.forward(x)
    four.forward_steps(x)
    torch().cuda.synchronize()
    moe.moe_check_device_status(one.ws)
    for name in ("topk_idx", "topk_w", "expert_offsets", "perm_token", "inv_slot", "y_perm", "y"):
        a, b = getattr(one, name), getattr(four, name)
        assert torch().equal(a, b), name


def test_layer_is_deterministic():
    cfg = synth.get_config("tiny", T=200, E=16, k=4, d=512, f=256)
    inp = synth.host_inputs(cfg)
    w = device_weights(cfg, inp)
    x = bf16_dev(inp.x)
    a = run_layer(cfg, x, w)
    ya, ia, pa = a.y.clone(), a.topk_idx.clone(), a.perm_token.clone()
    b = run_layer(cfg, x, w)
    assert torch().equal(ya.view(torch().int16), b.y.view(torch().int16))
    assert torch().equal(ia, b.topk_idx) and torch().equal(pa, b.perm_token)


@pytest.mark.parametrize("over", [{}, {"wdtype": "fp8", "T": 70, "E": 12, "k": 3, "d": 512, "f": 384},
                                  {"router": "zipf", "T": 600, "d": 512, "f": 256, "E": 16, "k": 2},
                                  {"wdtype": "mxfp4", "T": 600, "E": 8, "k": 2},
                                  {"T": 1100, "d": 512, "f": 256, "E": 128, "k": 4}])
def test_layer_replays_from_a_cuda_graph(over):
    # the four calls enqueue no synchronisation or allocation, so they can be captured once
    cfg = synth.get_config("tiny", **over)
    inp = synth.host_inputs(cfg)
    w = device_weights(cfg, inp)
    x = bf16_dev(inp.x)
    eager = run_layer(cfg, x, w).y.clone()
    layer = moe.MoeLayer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.n_shared, cfg.wdtype, w)
    layer.forward(x)
    torch().cuda.synchronize()
    g = torch().cuda.CUDAGraph()
    with torch().cuda.graph(g):
        layer.forward(x)
    layer.y.zero_()
    for _ in range(2):
        g.replay()
    torch().cuda.synchronize()
    moe.moe_check_device_status(layer.ws)
    assert torch().equal(eager.view(torch().int16), layer.y.view(torch().int16))


# ---- full-size workloads --------------------------------------------------------------------

def test_device_generator_matches_host_generator():
    cfg = synth.get_config("v3_decode")
    t = torch()
    n = 1 << 16
    buf = t.empty(n, dtype=t.bfloat16, device="cuda")
    for stream, sigma, off in ((synth.STREAM_X, 1.0, 12345), (synth.STREAM_W13, 0.02, 3 << 30)):
        synth._dev_normal(buf, cfg.seed, stream, sigma, offset=off)
        np.testing.assert_array_equal(bf16_host(buf), synth.normal_bf16(cfg.seed, stream, sigma, off, n))
    w = synth.normal_bf16(0, 4, 0.02, 777, 256 * 384).reshape(256, 384)
    q_h, s_h = synth.quantize_e4m3(w)
    q = t.empty(256, 384, dtype=t.uint8, device="cuda")
    s = t.empty(2, 3, dtype=t.float32, device="cuda")
    import ctypes
    rc = synth.lib().synth_quant_e4m3_device(bf16_dev(w).data_ptr(), q.data_ptr(), s.data_ptr(),
                                             256, 384, ctypes.c_void_p(t.cuda.current_stream().cuda_stream))
    assert rc == 0
    np.testing.assert_array_equal(q.cpu().numpy(), q_h)
    np.testing.assert_array_equal(s.cpu().numpy(), s_h)
    q4_h, s4_h = synth.quantize_mxfp4(w)
    q4 = t.empty(256, 192, dtype=t.uint8, device="cuda")
    s4 = t.empty(256, 12, dtype=t.uint8, device="cuda")
    rc = synth.lib().synth_quant_mxfp4_device(bf16_dev(w).data_ptr(), q4.data_ptr(), s4.data_ptr(),
                                              256, 384, ctypes.c_void_p(t.cuda.current_stream().cuda_stream))
    assert rc == 0
    np.testing.assert_array_equal(q4.cpu().numpy(), q4_h)
    np.testing.assert_array_equal(s4.cpu().numpy(), s4_h)


# The oracle decodes MXFP4 weights about 2.5x slower than E4M3 ones, so its full-size samples
# are smaller (the GPU suite stays within its time limit; the MXFP4 prefill tiles are the FP8
# kernel's, checked at the full FP8 sample).
def max_sampled_tokens(cfg):
    return 192 if cfg.wdtype == "mxfp4" else 512


def sample_tokens(cfg, idx, n_even=6):
    """Tokens whose outputs are checked in full. Below 1024 tokens: evenly spaced ones plus two
    tokens of the hottest and two of the coldest non-empty expert. From 1024 tokens: every
    s-th token (s = 8, or T/512 so that at most 512 tokens are checked; 192 for MXFP4 weights)
    plus two tokens of each of the four hottest and four coldest non-empty experts."""
    T = cfg.T
    counts = np.bincount(idx.ravel(), minlength=cfg.E)
    order = np.argsort(-counts, kind="stable")
    nonempty = [int(e) for e in order if counts[e] > 0]
    if T >= 1024:
        picks = set(range(0, T, max(8, T // max_sampled_tokens(cfg))))
        extremes = nonempty[:4] + nonempty[-4:]
    else:
        picks = set(np.linspace(0, T - 1, min(n_even, T)).astype(int).tolist())
        extremes = nonempty[:1] + nonempty[-1:]
    for e in extremes:
        rows = np.nonzero((idx == e).any(1))[0]
        picks.update(rows[:2].tolist())
    return sorted(picks)


FULL = ["v3_decode", "v4pro_decode", "skewed_prefill", "sweep_fp8_T1", "sweep_fp8_T8",
        "sweep_fp8_T64", "sweep_fp8_T256", "sweep_fp8_T1024", "sweep_fp8_T4096",
        "sweep_fp8_T16384", "v4pro_decode_fp4", "sweep_fp4_T1", "sweep_fp4_T8",
        "sweep_fp4_T64", "sweep_fp4_T256", "sweep_fp4_T1024", "sweep_fp4_T4096",
        "sweep_fp4_T16384"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_routing_exact_and_sampled_outputs(name):
    check_full(synth.get_config(name), name)


# The largest shapes the C ABI accepts along each axis: E = 1024 experts with k = 32 choices,
# d = 16384 (the longest router and gate/up reductions) and f = 16384 (the longest down one).
MAXIMUM = [
    {"T": 33, "d": 1024, "E": 1024, "k": 32, "f": 256},
    {"T": 5, "d": 16384, "E": 4, "k": 2, "f": 128},
    {"T": 5, "d": 128, "E": 4, "k": 2, "f": 16384},
    {"T": 5, "d": 16384, "E": 4, "k": 2, "f": 128, "wdtype": "fp8"},
    {"T": 5, "d": 128, "E": 4, "k": 2, "f": 16384, "wdtype": "fp8"},
    {"T": 5, "d": 16384, "E": 4, "k": 2, "f": 128, "wdtype": "mxfp4"},
    {"T": 5, "d": 128, "E": 4, "k": 2, "f": 16384, "wdtype": "mxfp4"},
]


@pytest.mark.parametrize("over", MAXIMUM, ids=[str(o) for o in MAXIMUM])
def test_maximum_shapes(over):
    check_full(synth.get_config("tiny", **over), "maximum " + str(over))


def weights_checksum(dev):
    """One int64 sum of every 32-bit word of the expert weights and scales (device-side): the
    layer must leave its inputs as they were."""
    t = torch()
    tot = 0
    for k in ("w13", "w2", "s13", "s2"):
        v = dev.get(k)
        if v is not None:
            tot += int(v.contiguous().view(t.int32).sum(dtype=t.int64).item())
    return tot


def device_expert(cfg, dev, e):
    """Expert e's weights as the seeded generator drew them on the device (the same bits as
    synth.host_expert, checked by test_device_generator_matches_host_generator), copied to the
    host. Drawing them on the host instead costs ~0.2 s an expert at the V3 shape."""
    t = torch()

    def h(v):
        if v is None:
            return None
        if v.dtype == t.bfloat16:
            return v[e].view(t.int16).cpu().numpy().view(np.uint16)
        return v[e].cpu().numpy()
    return synth.ExpertWeights(h(dev["w13"]), h(dev["w2"]), h(dev["s13"]), h(dev["s2"]))


def y_perm_rows_to_check(cfg, r_off, T):
    """Slots whose expert outputs are checked against the oracle: the last row of every routed
    expert that received tokens (each expert's weights, wherever they lie in HBM), the first and
    last rows of the shared segment, and from 1024 tokens every row of the four hottest and the
    four coldest non-empty experts (their deepest and shallowest token tiles; for MXFP4 weights
    the first 512 rows of each)."""
    counts = np.diff(r_off[: cfg.E + 1])
    rows = {int(r_off[e + 1]) - 1 for e in range(cfg.E) if counts[e] > 0}
    if cfg.n_shared and T > 0:
        rows.update({int(r_off[cfg.E]), int(r_off[cfg.E + 1]) - 1})
    if T >= 1024:
        order = [int(e) for e in np.argsort(-counts, kind="stable") if counts[e] > 0]
        cap = 512 if cfg.wdtype == "mxfp4" else 1 << 30
        for e in order[:4] + order[-4:]:
            rows.update(range(int(r_off[e]), min(int(r_off[e + 1]), int(r_off[e]) + cap)))
    return sorted(rows)


def check_y_perm_rows(cfg, layer, dev, x_h, r_off, r_perm, name):
    slots = y_perm_rows_to_check(cfg, r_off, cfg.T)
    routed = cfg.T * cfg.k
    by_expert = {}
    for s in slots:
        e = int(np.searchsorted(r_off[: cfg.E + 1], s, side="right") - 1) if s < routed else cfg.E
        by_expert.setdefault(e, []).append(s)
    yp = layer.y_perm
    worst = 0.0
    for e, ss in sorted(by_expert.items()):
        toks = [int(r_perm[s]) if s < routed else s - routed for s in ss]
        ew = device_expert(cfg, dev, e)
        ref = oracle.expert_rows(x_h[toks], ew.w13, ew.w2, cfg.wdtype, ew.s13, ew.s2)
        got = yp[ss].cpu().numpy().astype(np.float64)
        for r in range(len(ss)):
            rl = rel_l2(got[r], ref[r])
            worst = max(worst, rl)
            assert rl <= 1e-2, (name, "expert", e, "slot", ss[r], rl)
    return len(slots), worst


def router_uses_tc(cfg):
    return cfg.T >= 1024 and cfg.E % 128 == 0 and cfg.d % 64 == 0 and cfg.E <= 1024


def check_router_tc_logits(cfg, layer, x_h, wg_h, logits_nobias, name):
    """From 1024 tokens the router first forms every logit on the tensor cores (without the
    bias) into the workspace's logits area, and recomputes only the candidates in the defined
    order. Every one of the T*E approximate logits must lie within the bound the selection
    assumes, |a - l| <= 2^-12 |x_t| |wg_e|, of the defined fp32 logit l."""
    t = torch()
    n = cfg.T * cfg.E
    approx = layer.ws[256: 256 + 4 * n].view(t.float32).cpu().numpy().reshape(cfg.T, cfg.E)
    xf = oracle.bf16_to_f64(x_h)
    wf = oracle.bf16_to_f64(wg_h)
    bound = 2.0 ** -12 * np.outer(np.linalg.norm(xf, axis=1), np.linalg.norm(wf, axis=1))
    share = np.abs(approx.astype(np.float64) - logits_nobias.astype(np.float64)) / bound
    worst = float(share.max())
    assert worst <= 1.0, (name, "tensor-core logit outside its bound", worst)
    return worst


def check_full(cfg, name):
    dev = synth.device_inputs(cfg)
    w = {k: dev[k] for k in ("wg", "bias", "w13", "w2", "s13", "s2")}
    before = weights_checksum(dev)
    layer = run_layer(cfg, dev["x"], w)
    assert weights_checksum(dev) == before, "the layer changed its weights"
    idx = layer.topk_idx.cpu().numpy()
    # routing and permutation: every token, bit for bit
    x_h = synth.host_x(cfg)
    wg_h, bias_h = synth.host_wg(cfg), synth.host_bias(cfg)
    logits = oracle.router_logits(x_h, wg_h, bias_h)
    r_idx, _, r_w64 = oracle.route(logits, cfg.k)
    np.testing.assert_array_equal(idx, r_idx)
    np.testing.assert_allclose(layer.topk_w.cpu().numpy(), r_w64, rtol=0, atol=TOL_TOPK_W)
    r_off, r_perm, r_inv = oracle.permute(r_idx, cfg.E, cfg.n_shared)
    np.testing.assert_array_equal(layer.expert_offsets.cpu().numpy(), r_off)
    np.testing.assert_array_equal(layer.perm_token.cpu().numpy(), r_perm)
    np.testing.assert_array_equal(layer.inv_slot.cpu().numpy(), r_inv)
    # the tensor-core router's approximate logits, all T*E of them, within their bound
    if router_uses_tc(cfg):
        nob = logits if bias_h is None else oracle.router_logits(x_h, wg_h, None)
        share = check_router_tc_logits(cfg, layer, x_h, wg_h, nob, name)
        print(f"{name}: largest share of the router bound used by any logit {share:.3g}")
    # expert outputs (y_perm) of every expert that ran
    nrows, worst = check_y_perm_rows(cfg, layer, dev, x_h, r_off, r_perm, name)
    # outputs of sampled tokens, each straight from the definition
    toks = sample_tokens(cfg, r_idx)
    experts = {int(e): device_expert(cfg, dev, int(e)) for e in np.unique(r_idx[toks])}
    shared = device_expert(cfg, dev, cfg.E) if cfg.n_shared else None
    y_ref = oracle.token_outputs(x_h[toks], r_idx[toks], r_w64[toks], experts, shared, cfg.wdtype)
    y_gpu = bf16_host(layer.y)[toks]
    ma, rl = assert_y_close(y_gpu, y_ref, cfg.wdtype, what=name)
    print(f"{name}: {len(toks)} tokens (max-abs {ma:.3g}, rel-L2 {rl:.3g}), {nrows} expert "
          f"output rows (worst rel-L2 {worst:.3g})")


# ---- hash routing ----------------------------------------------------------------------------

def _hash_inputs(cfg, vocab=97):
    table = synth.hash_table(vocab, cfg.E, cfg.k, seed=cfg.seed)
    tid = synth.token_ids(cfg.T, vocab, seed=cfg.seed)
    return table, tid


@pytest.mark.parametrize("over", [{}, {"T": 300, "E": 40, "k": 5},
                                  {"T": 256, "d": 7168, "E": 256, "k": 8, "f": 128}])
def test_hash_route_matches_oracle(over):
    cfg = synth.get_config("tiny", **over)
    table, tid = _hash_inputs(cfg)
    x, wg, bias = synth.host_x(cfg), synth.host_wg(cfg), synth.host_bias(cfg)
    r_idx, _, r_w64 = oracle.route_hash(oracle.router_logits(x, wg, bias), tid, table)
    s = moe.shape_of(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.n_shared, cfg.wdtype)
    t = torch()
    ws = t.empty(moe.moe_workspace_size(s), dtype=t.uint8, device="cuda")
    idx = t.empty(cfg.T, cfg.k, dtype=t.int32, device="cuda")
    w = t.empty(cfg.T, cfg.k, dtype=t.float32, device="cuda")
    moe.moe_route_hash(s, bf16_dev(x), bf16_dev(wg), to_dev(bias), to_dev(tid), to_dev(table),
                       idx, w, ws)
    moe.moe_check_device_status(ws)
    np.testing.assert_array_equal(idx.cpu().numpy(), r_idx)
    np.testing.assert_allclose(w.cpu().numpy(), r_w64, rtol=0, atol=TOL_TOPK_W)


def test_hash_route_with_the_soft_choices_as_table_is_bit_identical_to_moe_route():
    cfg = synth.get_config("tiny", T=200, E=40, k=6)
    inp = synth.host_inputs(cfg)
    s = moe.shape_of(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.n_shared, cfg.wdtype)
    t = torch()
    ws = t.empty(moe.moe_workspace_size(s), dtype=t.uint8, device="cuda")
    idx = t.empty(cfg.T, cfg.k, dtype=t.int32, device="cuda")
    w = t.empty(cfg.T, cfg.k, dtype=t.float32, device="cuda")
    x, wg = bf16_dev(inp.x), bf16_dev(inp.wg)
    moe.moe_route(s, x, wg, None, idx, w, ws)
    hidx, hw = t.empty_like(idx), t.empty_like(w)
    moe.moe_route_hash(s, x, wg, None, t.arange(cfg.T, dtype=t.int32, device="cuda"), idx.clone(),
                       hidx, hw, ws)
    moe.moe_check_device_status(ws)
    assert t.equal(hidx, idx) and t.equal(hw.view(t.int32), w.view(t.int32))


@pytest.mark.parametrize("over", [{}, {"wdtype": "fp8"}, {"wdtype": "mxfp4"},
                                  {"T": 300, "E": 40, "k": 5, "d": 512, "f": 256}])
def test_hash_routed_layer_matches_oracle(over):
    cfg = synth.get_config("tiny", **over)
    inp = synth.host_inputs(cfg)
    table, tid = _hash_inputs(cfg)
    w = device_weights(cfg, inp)
    layer = moe.MoeLayer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.n_shared, cfg.wdtype, w)
    layer.forward_hash(bf16_dev(inp.x), to_dev(tid), to_dev(table))
    torch().cuda.synchronize()
    moe.moe_check_device_status(layer.ws)
    r_idx, _, r_w64 = oracle.route_hash(oracle.router_logits(inp.x, inp.wg, inp.bias), tid, table)
    np.testing.assert_array_equal(layer.topk_idx.cpu().numpy(), r_idx)
    r_off, r_perm, r_inv = oracle.permute(r_idx, cfg.E, cfg.n_shared)
    np.testing.assert_array_equal(layer.expert_offsets.cpu().numpy(), r_off)
    np.testing.assert_array_equal(layer.perm_token.cpu().numpy(), r_perm)
    experts = {e: inp.experts[e] for e in range(cfg.E)}
    shared = inp.experts[cfg.E] if cfg.n_shared else None
    y_ref = oracle.token_outputs(inp.x, r_idx, r_w64, experts, shared, cfg.wdtype)
    assert_y_close(bf16_host(layer.y), y_ref, cfg.wdtype, what="hash-routed layer")


def test_hash_route_flags_bad_token_id_and_table_entry_without_faulting():
    cfg = synth.get_config("tiny")
    table, tid = _hash_inputs(cfg)
    s = moe.shape_of(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.n_shared, cfg.wdtype)
    t = torch()
    ws = t.empty(moe.moe_workspace_size(s), dtype=t.uint8, device="cuda")
    idx = t.empty(cfg.T, cfg.k, dtype=t.int32, device="cuda")
    w = t.empty(cfg.T, cfg.k, dtype=t.float32, device="cuda")
    x, wg = bf16_dev(synth.host_x(cfg)), bf16_dev(synth.host_wg(cfg))
    for bad_tid, bad_table in ((True, False), (False, True)):
        tid_b, table_b = tid.copy(), table.copy()
        if bad_tid:
            tid_b[3] = table.shape[0]          # one past the last row
        else:
            table_b[tid[5], 1] = cfg.E          # an expert that does not exist
        moe.moe_route_hash(s, x, wg, None, to_dev(tid_b), to_dev(table_b), idx, w, ws)
        with pytest.raises(moe.MoeError) as err:
            moe.moe_check_device_status(ws)
        assert err.value.status == -6
        assert np.all((idx.cpu().numpy() >= 0) & (idx.cpu().numpy() < cfg.E))
    # the context is still usable: a clean call passes its check
    moe.moe_route_hash(s, x, wg, None, to_dev(tid), to_dev(table), idx, w, ws)
    moe.moe_check_device_status(ws)
