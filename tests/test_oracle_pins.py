"""Pins of the CPU oracle to facts outside itself: the pages' worked examples, format
definitions, library-routine reductions, brute force and invariants."""
import math

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle
import synth
from conftest import golden_kv, golden_rows


def bf16_bits(vals):
    """Exact bf16 bit patterns of values that bf16 represents exactly."""
    f = np.asarray(vals, dtype=np.float32)
    b = f.view(np.uint32)
    assert np.all(b & 0xFFFF == 0), "value not exactly representable in bf16"
    return (b >> 16).astype(np.uint16)


def rand_bf16(rng, shape, sigma=1.0):
    return synth.double_to_bf16(rng.normal(0.0, sigma, size=shape))


# ---- worked example: "第 6 章 超節點", 6.2.2 ----------------------------------------------------

def test_worked_example_matvec_and_splits():
    g = golden_kv("matmul_split_2x2.txt")
    x = np.array([float(v) for v in g["x"].split()])
    W = np.array([[float(v) for v in g["W_row0"].split()], [float(v) for v in g["W_row1"].split()]])
    Wt = bf16_bits(W.T.copy())  # stored [out, in]
    np.testing.assert_array_equal(oracle.matvec(Wt, x), [float(v) for v in g["xW"].split()])
    # column split: each device computes its own output features
    assert oracle.matvec(Wt, x, row0=0, nrows=1)[0] == float(g["col_split_0"])
    assert oracle.matvec(Wt, x, row0=1, nrows=1)[0] == float(g["col_split_1"])
    # row split: each device sees part of the input features, outputs are partial sums
    p0 = oracle.matvec(Wt, np.array([x[0], 0.0]))
    p1 = oracle.matvec(Wt, np.array([0.0, x[1]]))
    np.testing.assert_array_equal(p0, [float(v) for v in g["row_split_0"].split()])
    np.testing.assert_array_equal(p1, [float(v) for v in g["row_split_1"].split()])
    np.testing.assert_array_equal(p0 + p1, [float(v) for v in g["xW"].split()])


def test_fp8_block_scales_index_by_row_and_column_block():
    # 256 x 256 E4M3 matrix of code 0x38 (1.0) with a different scale in each 128x128 block:
    # with a one-hot x, W x picks out column c, whose entries are 1.0 * s[r//128][c//128].
    q = np.full((256, 256), 0x38, dtype=np.uint8)
    s = np.array([[2.0, 3.0], [5.0, 7.0]], dtype=np.float32)
    for c, expect in ((0, [2.0, 5.0]), (200, [3.0, 7.0])):
        x = np.zeros(256)
        x[c] = 1.0
        y = oracle.matvec(q, x, wdtype="fp8", s=s)
        np.testing.assert_array_equal(y[:128], expect[0])
        np.testing.assert_array_equal(y[128:], expect[1])


# ---- number formats -----------------------------------------------------------------------

def test_e4m3_decode_golden_codes():
    for row in golden_rows("e4m3_codes.txt"):
        code, val = row.split()
        v = oracle.e4m3_value(int(code, 16))
        if val == "nan":
            assert math.isnan(v)
        else:
            assert v == float(val) and math.copysign(1.0, v) == math.copysign(1.0, float(val))


def test_e4m3_decode_roundtrips_through_the_independent_encoder():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = np.array([oracle.e4m3_value(int(c)) for c in codes], dtype=np.float32)
    back = synth.f32_to_e4m3(vals)
    # +0 and -0 both decode to zero; everything else must map back to its own code
    np.testing.assert_array_equal(back, codes)
    assert np.all(np.diff(vals[(codes < 0x80)]) > 0)  # positive codes are strictly increasing


def test_mxfp4_element_and_scale_decode_golden_codes():
    for row in golden_rows("mxfp4_codes.txt"):
        kind, code, val = row.split()
        v = (oracle.e2m1_value if kind == "e2m1" else oracle.e8m0_value)(int(code, 16))
        if val == "nan":
            assert math.isnan(v)
        else:
            assert v == float(val) and math.copysign(1.0, v) == math.copysign(1.0, float(val))


def mxfp4_reference_quantise(w: np.ndarray):
    """The OCP MX quantisation of fp64 weights [rows, cols], restated in numpy: per 32
    consecutive elements of a row, X = 2^(floor(log2 amax) - 2), element = the nearest of the
    E2M1 magnitudes to |w|/X (ties to the one with mantissa bit 0), saturating at 6. Returns
    the dequantised fp64 weights."""
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    rows, cols = w.shape
    b = w.reshape(rows, cols // 32, 32)
    amax = np.abs(b).max(axis=2, keepdims=True)
    with np.errstate(divide="ignore"):
        X = np.where(amax > 0, 2.0 ** (np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2), 1.0)
    a = np.abs(b) / X
    dist = np.abs(a[..., None] - grid)
    best = dist.min(axis=-1, keepdims=True)
    cand = np.isclose(dist, best, rtol=0, atol=0)
    # among equally near magnitudes take the even code (index 0, 2, 4, 6)
    even = cand & (np.arange(8) % 2 == 0)
    pick = np.where(even.any(-1), even.argmax(-1), cand.argmax(-1))
    return (np.sign(b) * grid[pick] * X).reshape(rows, cols)


def test_mxfp4_quantise_then_decode_matches_numpy_restatement():
    rng = np.random.default_rng(5)
    w = rand_bf16(rng, (64, 256), sigma=0.02)
    # a zero block, a block with a tie at every grid midpoint, and a saturating block
    w[0, :32] = 0
    w[1, :32] = bf16_bits(np.resize([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 4.0], 32))
    w[2, :32] = bf16_bits(np.resize([7.5, -7.5, 4.0, 1.0], 32))
    q, s = synth.quantize_mxfp4(w)
    deq = np.array([[oracle.matvec(q, np.eye(256)[c], "mxfp4", s, row0=r, nrows=1)[0]
                     for c in range(256)] for r in range(4)])
    ref = mxfp4_reference_quantise(oracle.bf16_to_f64(w))
    np.testing.assert_array_equal(deq, ref[:4])
    # the rest through the layer's own matvec: W x with x = all ones is each row's sum
    np.testing.assert_allclose(oracle.matvec(q, np.ones(256), "mxfp4", s), ref.sum(1),
                               rtol=1e-14, atol=1e-14)


def test_mxfp4_scales_index_by_row_and_32_column_block_and_low_nibble_first():
    # every element code 0x2 (1.0) except element 1 of each row (code 0x4, 2.0): byte 0 is 0x42
    rows, cols = 4, 96
    q = np.full((rows, cols // 2), 0x22, np.uint8)
    q[:, 0] = 0x42
    s = (127 + np.arange(rows * 3).reshape(rows, 3)).astype(np.uint8)  # 2^(3r + j)
    for c in (0, 1, 40, 95):
        x = np.zeros(cols)
        x[c] = 1.0
        elem = 2.0 if c == 1 else 1.0
        expect = [elem * 2.0 ** (3 * r + c // 32) for r in range(rows)]
        np.testing.assert_array_equal(oracle.matvec(q, x, "mxfp4", s), expect)


def test_bf16_decode():
    assert oracle.bf16_value(0x3F80) == 1.0
    assert oracle.bf16_value(0xC000) == -2.0
    assert oracle.bf16_value(0x3B80) == 2.0 ** -8
    assert oracle.bf16_value(0x0001) == 2.0 ** -133  # smallest subnormal
    assert oracle.bf16_value(0x7F7F) == (2 - 2 ** -7) * 2.0 ** 127


# ---- a1: router ---------------------------------------------------------------------------

def _parse(v):
    v = v.strip()
    if v == "1+2^-23":
        return 1.0 + 2.0 ** -23
    if v.startswith("2^"):
        return 2.0 ** float(v[2:])
    return float(v)


def test_router_logit_fixed_order_cases():
    for row in golden_rows("router_logit_order.txt"):
        name, d, prods, expect = (c.strip() for c in row.split("|"))
        d = int(d)
        x, w = np.zeros(d, np.float32), np.zeros(d, np.float32)
        for p in prods.split():
            i, xv, wv = p.split(":")
            x[int(i)], w[int(i)] = _parse(xv), _parse(wv)
        l = oracle.router_logits(bf16_bits(x)[None, :], bf16_bits(w)[None, :])
        assert l[0, 0] == np.float32(_parse(expect)), name


def test_router_logit_bias_is_added_after_the_dot_product():
    x = bf16_bits(np.array([1.0] + [0.0] * 255))[None, :]
    w = bf16_bits(np.array([[0.5] + [0.0] * 255, [0.25] + [0.0] * 255]))
    l = oracle.router_logits(x, w, np.array([1.0, -3.0], np.float32))
    np.testing.assert_array_equal(l, [[1.5, -2.75]])


def test_router_logits_within_fp32_error_bound_of_exact_sum():
    rng = np.random.default_rng(1)
    T, d, E = 3, 7168, 5
    x, wg = rand_bf16(rng, (T, d)), rand_bf16(rng, (E, d), 0.02)
    l = oracle.router_logits(x, wg)
    xf, wf = oracle.bf16_to_f64(x), oracle.bf16_to_f64(wg)
    n = d // 32 + 5
    gamma = n * 2.0 ** -24 / (1 - n * 2.0 ** -24)
    for t in range(T):
        for e in range(E):
            prods = xf[t] * wf[e]                 # exact in fp64
            exact = math.fsum(prods)
            assert abs(float(l[t, e]) - exact) <= gamma * np.abs(prods).sum()


def _routing_case(seed=2, T=40, E=24, d=256):
    rng = np.random.default_rng(seed)
    return oracle.router_logits(rand_bf16(rng, (T, d)), rand_bf16(rng, (E, d), 0.02))


@pytest.mark.parametrize("k", [1, 3, 8, 24])
def test_topk_matches_full_sort(k):
    l = _routing_case()
    idx, w, w64 = oracle.route(l, k)
    T, E = l.shape
    for t in range(T):
        order = np.lexsort((np.arange(E), -l[t].astype(np.float64)))  # logit desc, index asc
        np.testing.assert_array_equal(idx[t], order[:k])


def test_topk_weights_k_equals_E_is_full_softmax_and_k1_is_one():
    l = _routing_case()
    T, E = l.shape
    idx, _, w64 = oracle.route(l, E)
    for t in range(T):
        full = softmax(l[t].astype(np.float64))
        np.testing.assert_allclose(w64[t], full[idx[t]], rtol=1e-13, atol=0)
    _, w1, w164 = oracle.route(l, 1)
    assert np.all(w1 == 1.0) and np.all(w164 == 1.0)


def test_topk_weights_sum_to_one_and_equal_softmax_over_chosen():
    l = _routing_case()
    idx, w, w64 = oracle.route(l, 6)
    np.testing.assert_allclose(w64.sum(1), 1.0, atol=1e-14)
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= 1e-6)
    for t in range(l.shape[0]):
        np.testing.assert_allclose(w64[t], softmax(l[t, idx[t]].astype(np.float64)), rtol=1e-13)


def test_hash_route_with_the_soft_choices_as_table_is_the_soft_route():
    # a table that holds, for each token id, exactly the soft router's choice: both routes agree
    rng = np.random.default_rng(11)
    T, E, k = 40, 24, 5
    logits = rng.normal(size=(T, E)).astype(np.float32)
    idx, w, w64 = oracle.route(logits, k)
    h_idx, h_w, h_w64 = oracle.route_hash(logits, np.arange(T, dtype=np.int32), idx)
    np.testing.assert_array_equal(h_idx, idx)
    np.testing.assert_array_equal(h_w, w)
    np.testing.assert_allclose(h_w64, w64, rtol=1e-15, atol=0)


def test_hash_route_weights_are_the_softmax_of_the_hashed_logits():
    rng = np.random.default_rng(12)
    T, E, k, vocab = 33, 16, 4, 50
    logits = rng.normal(size=(T, E)).astype(np.float32) * 3
    table = np.stack([rng.permutation(E)[:k] for _ in range(vocab)]).astype(np.int32)
    tid = rng.integers(0, vocab, T).astype(np.int32)
    idx, _, w64 = oracle.route_hash(logits, tid, table)
    np.testing.assert_array_equal(idx, table[tid])  # the table's experts, in its order
    chosen = np.take_along_axis(logits.astype(np.float64), table[tid], axis=1)
    np.testing.assert_allclose(w64, softmax(chosen, axis=1), rtol=1e-12, atol=0)
    # k = 1: the one hashed expert gets weight 1
    _, _, w1 = oracle.route_hash(logits, tid, table[:, :1])
    np.testing.assert_array_equal(w1, 1.0)


def test_topk_ties_go_to_lower_index():
    x = rand_bf16(np.random.default_rng(3), (4, 256))
    row = rand_bf16(np.random.default_rng(4), (1, 256), 0.02)
    wg = np.repeat(row, 8, axis=0)                 # eight identical experts -> equal logits
    idx, w, _ = oracle.route(oracle.router_logits(x, wg), 3)
    np.testing.assert_array_equal(idx, np.tile([0, 1, 2], (4, 1)))
    np.testing.assert_allclose(w, 1.0 / 3.0, rtol=1e-7)


def test_distinct_experts_hit_matches_eq_6_8_within_5_percent():
    # plain router on the V3 shape: E=256, k=8, m=64 tokens -> eq. 6-8 expects 222.6 experts
    cfg = synth.get_config("v3_decode", T=64)
    l = oracle.router_logits(synth.host_x(cfg), synth.host_wg(cfg))
    idx, _, _ = oracle.route(l, cfg.k)
    expect = cfg.E * (1 - (1 - cfg.k / cfg.E) ** cfg.T)
    assert abs(len(np.unique(idx)) - expect) <= 0.05 * expect


# ---- a2: permutation ------------------------------------------------------------------------

def _random_topk(rng, T, E, k):
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k,S", [(37, 8, 2, 1), (64, 16, 16, 1), (5, 1, 1, 0), (0, 4, 2, 1),
                                     (100, 33, 3, 0)])
def test_permutation_is_stable_counting_sort(T, E, k, S):
    rng = np.random.default_rng(T + E)
    idx = _random_topk(rng, T, E, k) if T else np.zeros((0, k), np.int32)
    off, perm, inv = oracle.permute(idx, E, S)
    counts = np.bincount(idx.ravel(), minlength=E)
    np.testing.assert_array_equal(np.diff(off[: E + 1]), counts)
    assert off[0] == 0 and off[E] == T * k and off[E + 1] == T * k + S * T
    # brute force: stable sort of (expert, token) pairs
    tok = np.repeat(np.arange(T), k)
    order = np.lexsort((tok, idx.ravel()))
    np.testing.assert_array_equal(perm, tok[order])
    pos = np.empty(T * k, np.int64)
    pos[order] = np.arange(T * k)
    np.testing.assert_array_equal(inv, pos)
    # invariants
    if T:
        np.testing.assert_array_equal(perm[inv], tok)
        np.testing.assert_array_equal(np.bincount(perm, minlength=T), np.full(T, k))


# ---- a3 + a4: SwiGLU expert ------------------------------------------------------------------

def test_swiglu_known_values_gate_then_up_then_down():
    # x = one-hot, gate/up weights hold chosen scalars in column 0, W_d routes h_r to y_r:
    # then y_r = SiLU(g_r) * u_r with SiLU(z) = z * logistic(z).
    d, f = 128, 128
    g = np.array([0.0, 2.0, -2.0, 8.0, 0.5, -0.25] + [1.0] * (f - 6))
    u = np.array([3.0, 1.0, 1.0, 0.5, -2.0, 4.0] + [0.0] * (f - 6))
    w13 = np.zeros((2 * f, d), np.float32)
    w13[:f, 0], w13[f:, 0] = g, u
    w2 = np.eye(d, f, dtype=np.float32)
    x = np.zeros((1, d), np.float32)
    x[0, 0] = 1.0
    y, h = oracle.expert_rows(bf16_bits(x), bf16_bits(w13), bf16_bits(w2), want_h=True)
    np.testing.assert_allclose(h[0], g * expit(g) * u, rtol=1e-15, atol=1e-300)
    np.testing.assert_allclose(y[0], h[0], rtol=0, atol=0)


def test_swiglu_split_intermediate_sums_eq_6_3():
    # Y = Z0 Wd0 + Z1 Wd1 when the intermediate width f is split in two halves.
    rng = np.random.default_rng(5)
    d, f = 128, 256
    x = rand_bf16(rng, (3, d))
    w13, w2 = rand_bf16(rng, (2 * f, d), 0.02), rand_bf16(rng, (d, f), 0.02)
    full = oracle.expert_rows(x, w13, w2)
    half = f // 2
    parts = []
    for s in (slice(0, half), slice(half, f)):
        w13_s = np.concatenate([w13[:f][s], w13[f:][s]])
        parts.append(oracle.expert_rows(x, w13_s, np.ascontiguousarray(w2[:, s])))
    np.testing.assert_allclose(parts[0] + parts[1], full, rtol=1e-12, atol=1e-15)


def test_single_expert_layer_is_a_dense_swiglu_ffn():
    # E = 1, k = 1, no shared expert: the layer is Y = [SiLU(X Wg) (.) (X Wu)] Wd (numpy matmul).
    cfg = synth.get_config("tiny", E=1, k=1, n_shared=0, T=9)
    inp = synth.host_inputs(cfg)
    out = oracle.moe_layer(cfg, inp)
    X = oracle.bf16_to_f64(inp.x)
    W13 = oracle.bf16_to_f64(inp.experts[0].w13)
    Wd = oracle.bf16_to_f64(inp.experts[0].w2)
    G, U = X @ W13[: cfg.f].T, X @ W13[cfg.f:].T
    Y = (G * expit(G) * U) @ Wd.T
    np.testing.assert_allclose(out["y"], Y, rtol=1e-11, atol=1e-13)
    assert np.all(out["topk_idx"] == 0) and np.all(out["topk_w"] == 1.0)


def dense_expert_outputs(cfg, inp):
    """Every expert's SwiGLU output for every token, [E + n_shared, T, d], with numpy from the
    format definitions (E4M3 codes by the oracle's golden-pinned decoder, E2M1 by its formula)."""
    X = oracle.bf16_to_f64(inp.x)

    def dense_w(ew, which):
        if cfg.wdtype == "bf16":
            return oracle.bf16_to_f64(getattr(ew, which))
        q = getattr(ew, which)
        s = getattr(ew, "s" + which[1:])
        if cfg.wdtype == "mxfp4":
            # the E2M1 magnitudes by the format's formula, both nibbles, times 2^(e-127)
            codes = np.stack([q & 15, q >> 4], axis=-1).reshape(q.shape[0], -1)
            mag = np.where((codes >> 1) & 3 == 0, 0.5 * (codes & 1),
                           2.0 ** (((codes >> 1) & 3).astype(int) - 1) * (1 + 0.5 * (codes & 1)))
            X_ = np.repeat(2.0 ** (s.astype(int) - 127), 32, axis=1)
            return np.where(codes & 8, -1.0, 1.0) * mag * X_
        vals = np.array([oracle.e4m3_value(c) for c in range(256)])[q]
        return vals * np.kron(s.astype(np.float64), np.ones((128, 128)))

    Ys = []
    for ew in inp.experts:
        W13, Wd = dense_w(ew, "w13"), dense_w(ew, "w2")
        G, U = X @ W13[: cfg.f].T, X @ W13[cfg.f:].T
        Ys.append((G * expit(G) * U) @ Wd.T)
    return np.stack(Ys)


def dense_masked_layer(cfg, Ys, topk_idx, topk_w64):
    """y = shared + sum over experts of (gate weight, 0 if not chosen) x expert output."""
    mask = np.zeros((cfg.T, cfg.E))
    for t in range(cfg.T):
        mask[t, topk_idx[t]] = topk_w64[t]
    y = np.einsum("te,etd->td", mask, Ys[: cfg.E])
    if cfg.n_shared:
        y += Ys[cfg.E]
    return y


@pytest.mark.parametrize("name,over", [("tiny", {}), ("tiny", {"wdtype": "fp8"}),
                                       ("tiny", {"wdtype": "mxfp4"}),
                                       ("tiny", {"n_shared": 0, "k": 3}),
                                       ("tiny", {"router": "zipf", "T": 21})])
def test_layer_equals_dense_masked_evaluation(name, over):
    # every expert evaluated on every token with numpy, non-chosen ones weighted 0
    cfg = synth.get_config(name, **over)
    inp = synth.host_inputs(cfg)
    out = oracle.moe_layer(cfg, inp)
    y = dense_masked_layer(cfg, dense_expert_outputs(cfg, inp), out["topk_idx"], out["topk_w64"])
    np.testing.assert_allclose(out["y"], y, rtol=1e-10, atol=1e-14)


# ---- token_outputs: y of a sample of tokens, as the full-size GPU checks use it ----------------

TOKEN_OUTPUT_CASES = [("tiny", {}), ("tiny", {"wdtype": "fp8"}), ("tiny", {"wdtype": "mxfp4"}),
                      ("tiny", {"n_shared": 0}), ("tiny", {"n_shared": 0, "wdtype": "fp8"}),
                      ("tiny", {"router": "zipf", "T": 45}), ("tiny", {"k": 8}),
                      ("tiny", {"T": 1}), ("tiny", {"T": 1, "wdtype": "mxfp4", "k": 3})]


@pytest.mark.parametrize("name,over", TOKEN_OUTPUT_CASES, ids=[str(o) for _, o in TOKEN_OUTPUT_CASES])
def test_token_outputs_equal_the_whole_layer(name, over):
    # "第 6 章 超節點", 6.2.6: a token's output is the gate-weighted sum of its experts' outputs
    # (a1 y1 + a6 y6), plus the always-on shared expert. token_outputs forms it per token from
    # the routing; it must equal the whole layer's y (pinned to the dense masked evaluation
    # above) for all tokens, and for a subset given in a scrambled order.
    cfg = synth.get_config(name, **over)
    inp = synth.host_inputs(cfg)
    out = oracle.moe_layer(cfg, inp)
    experts = {e: inp.experts[e] for e in range(cfg.E)}
    shared = inp.experts[cfg.E] if cfg.n_shared else None
    for toks in (list(range(cfg.T)), list(range(cfg.T - 1, -1, -3))):
        y = oracle.token_outputs(inp.x[toks], out["topk_idx"][toks], out["topk_w64"][toks],
                                 experts, shared, cfg.wdtype)
        np.testing.assert_allclose(y, out["y"][toks], rtol=0, atol=1e-12)


@pytest.mark.parametrize("wdtype", ["bf16", "fp8"])
def test_token_outputs_of_hash_routing_equal_the_dense_masked_evaluation(wdtype):
    cfg = synth.get_config("tiny", T=30, k=3, wdtype=wdtype)
    inp = synth.host_inputs(cfg)
    table = synth.hash_table(41, cfg.E, cfg.k, seed=3)
    tid = synth.token_ids(cfg.T, 41, seed=3)
    idx, _, w64 = oracle.route_hash(oracle.router_logits(inp.x, inp.wg, inp.bias), tid, table)
    y_ref = dense_masked_layer(cfg, dense_expert_outputs(cfg, inp), idx, w64)
    y = oracle.token_outputs(inp.x, idx, w64, {e: inp.experts[e] for e in range(cfg.E)},
                             inp.experts[cfg.E], cfg.wdtype)
    np.testing.assert_allclose(y, y_ref, rtol=1e-10, atol=1e-14)


# ---- a5: combine ----------------------------------------------------------------------------

def test_combine_four_contributions_sum_to_ten():
    g = golden_kv("combine_sum.txt")
    w = np.array([[float(v) for v in g["weights"].split()]])
    idx = np.array([[0, 1, 2, 3]], np.int32)
    off, perm, inv = oracle.permute(idx, 4, 0)
    y_perm = np.full((4, 3), float(g["expert_output"]))
    y = oracle.combine(y_perm, inv, w, 1, 4, n_shared=0)
    np.testing.assert_allclose(y, float(g["expected"]), rtol=1e-15)


def test_combine_is_a1_y1_plus_a6_y6_plus_shared():
    rng = np.random.default_rng(7)
    idx = np.array([[6, 1], [3, 6]], np.int32)          # token A -> experts 6 and 1
    w = np.array([[0.7, 0.3], [0.55, 0.45]])
    off, perm, inv = oracle.permute(idx, 8, 1)
    y_perm = rng.normal(size=(off[-1], 5))
    y = oracle.combine(y_perm, inv, w, 2, 2, n_shared=1)
    slot = {(int(perm[s]), e): s for e in range(8) for s in range(off[e], off[e + 1])}
    a6, a1 = w[0]
    y1, y6, shared = y_perm[slot[(0, 1)]], y_perm[slot[(0, 6)]], y_perm[4 + 0]
    np.testing.assert_allclose(y[0], a1 * y1 + a6 * y6 + shared, rtol=1e-15)
