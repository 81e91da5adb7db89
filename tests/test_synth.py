"""The seeded input generator: determinism, slicing, distributions, FP8 quantiser, workloads."""
import numpy as np
import pytest

import oracle
import synth


def test_stream_slices_are_consistent_and_deterministic():
    a = synth.normal_bf16(0, 3, 0.02, 0, 5000)
    b = synth.normal_bf16(0, 3, 0.02, 1234, 100)
    np.testing.assert_array_equal(a[1234:1334], b)
    np.testing.assert_array_equal(a, synth.normal_bf16(0, 3, 0.02, 0, 5000))
    assert not np.array_equal(a, synth.normal_bf16(1, 3, 0.02, 0, 5000))
    assert not np.array_equal(a, synth.normal_bf16(0, 4, 0.02, 0, 5000))


def test_normal_moments_and_bounds():
    v = oracle.bf16_to_f64(synth.normal_bf16(0, 1, 1.0, 0, 1 << 20))
    assert abs(v.mean()) < 0.005 and abs(v.std() - 1.0) < 0.005
    assert np.abs(v).max() <= 6.0
    # Irwin-Hall(12) kurtosis is 3 - 1.2/12 = 2.9
    assert abs(((v - v.mean()) ** 4).mean() / v.var() ** 2 - 2.9) < 0.03
    w = oracle.bf16_to_f64(synth.normal_bf16(0, 3, 0.02, 0, 1 << 18))
    assert abs(w.std() - 0.02) < 0.0003


def test_double_to_bf16_round_to_nearest_even():
    one = 1.0
    ulp = 2.0 ** -7
    cases = [(one, 0x3F80), (one + ulp / 2, 0x3F80), (one + 1.5 * ulp, 0x3F82),
             (one + ulp / 2 + 1e-12, 0x3F81), (-2.0, 0xC000), (0.0, 0x0000),
             (2.0 ** -133, 0x0001), (3.5e38, 0x7F80)]
    got = synth.double_to_bf16(np.array([c for c, _ in cases]))
    np.testing.assert_array_equal(got, [b for _, b in cases])


def test_f32_to_e4m3_rounding_and_saturation():
    vals = np.array([1.0, 1.0625, 1.1875, 448.0, 500.0, 1e9, -1e9, 2.0 ** -10, 3 * 2.0 ** -10,
                     -0.0, 0.0], np.float32)
    # 1.0625 is halfway 1.0/1.125 -> even (1.0); 1.1875 halfway 1.125/1.25 -> 1.25 (even)
    expect = [0x38, 0x38, 0x3A, 0x7E, 0x7E, 0x7E, 0xFE, 0x00, 0x02, 0x80, 0x00]
    np.testing.assert_array_equal(synth.f32_to_e4m3(vals), expect)


def test_quantiser_block_scale_and_error_bound():
    w = synth.normal_bf16(0, 3, 0.02, 0, 256 * 384).reshape(256, 384)
    q, s = synth.quantize_e4m3(w)
    wf = oracle.bf16_to_f64(w)
    deq = np.array([oracle.e4m3_value(c) for c in range(256)])[q] * np.kron(s, np.ones((128, 128)))
    for rb in range(2):
        for cb in range(3):
            blk = wf[rb * 128:(rb + 1) * 128, cb * 128:(cb + 1) * 128]
            assert s[rb, cb] == np.float32(np.float32(np.abs(blk).max()) / np.float32(448.0))
    # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 for normals, abs <= s*2^-10 subnormals
    err = np.abs(deq - wf)
    bound = np.maximum(np.abs(wf) * 2.0 ** -4, np.kron(s, np.ones((128, 128))) * 2.0 ** -10)
    assert np.all(err <= bound * (1 + 1e-6))


def test_zipf_bias_is_a_permuted_power_law():
    b = synth.zipf_bias(256, 0)
    ranks = np.argsort(-b)
    z = np.exp(b.astype(np.float64) / 1.5)
    np.testing.assert_allclose(z.sum(), 1.0, rtol=1e-5)
    zs = z[ranks]
    np.testing.assert_allclose(zs[1:] / zs[0], np.arange(2, 257) ** -1.1, rtol=1e-4)
    assert sorted(ranks.tolist()) == list(range(256)) and ranks[0] != 0


def test_skewed_prefill_workload_is_skewed():
    # The Zipf workload must give a few hot experts (>1000 tokens) and many cold ones (<8).
    # Counts from an fp32 numpy router are enough for this property of the inputs.
    cfg = synth.get_config("skewed_prefill")
    x = oracle.bf16_to_f64(synth.host_x(cfg)).astype(np.float32)
    wg = oracle.bf16_to_f64(synth.host_wg(cfg)).astype(np.float32)
    logits = x @ wg.T + synth.host_bias(cfg)
    top = np.argsort(-logits, axis=1)[:, : cfg.k]
    counts = np.bincount(top.ravel(), minlength=cfg.E)
    assert counts.max() > 1000 and (counts < 8).sum() >= 64


def test_configs():
    for name in ("tiny", "v3_decode", "v4pro_decode", "skewed_prefill", "sweep_fp8_T16384"):
        c = synth.get_config(name)
        assert c.d % 128 == 0 and c.f % 128 == 0 and 1 <= c.k <= c.E
    c = synth.get_config("v4pro_decode")
    assert (c.T, c.E, c.k, c.f, c.wdtype) == (32, 384, 6, 3072, "fp8")
    with pytest.raises(KeyError):
        synth.get_config("nope")


def test_f32_to_e2m1_rounding_ties_and_saturation():
    v = np.array([0.0, 0.24, 0.25, 0.26, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 5.01, 6.0, 100.0,
                  -0.75, -5.01], np.float32)
    # magnitude codes 0..7 are 0, 0.5, 1, 1.5, 2, 3, 4, 6; ties go to the even code
    expect = [0, 0, 0, 1, 2, 2, 4, 4, 6, 6, 7, 7, 7, 0x8 | 2, 0x8 | 7]
    np.testing.assert_array_equal(synth.f32_to_e2m1(v), expect)


def test_mxfp4_quantiser_scale_rule_and_layout():
    rng = np.random.default_rng(3)
    w = synth.double_to_bf16(rng.normal(0.0, 0.02, size=(8, 128)))
    q, s = synth.quantize_mxfp4(w)
    assert q.shape == (8, 64) and s.shape == (8, 4)
    f = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(8, 4, 32)
    amax = np.abs(f).max(2)
    np.testing.assert_array_equal(s, np.floor(np.log2(amax)).astype(int) - 2 + 127)
    # element 2j in the low nibble: decode both nibbles by the E2M1 formula and rebuild
    mag = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    codes = np.stack([q & 15, q >> 4], axis=-1).reshape(8, 128)
    vals = np.where(codes & 8, -1.0, 1.0) * mag[codes & 7]
    X = np.repeat(2.0 ** (s.astype(int) - 127), 32, axis=1)
    err = np.abs(vals * X - f.reshape(8, 128))
    # within half a step of E2M1 at the element's magnitude (steps 0.5, 1, 2 by binade), or a
    # saturation at 6 of a value below 8
    half_step = np.where(np.abs(f.reshape(8, 128)) / X < 2, 0.25, np.where(np.abs(f.reshape(8, 128)) / X < 4, 0.5, 1.0)) * X
    assert np.all((err <= half_step) | (np.abs(vals) == 6.0))


def test_hash_table_rows_are_distinct_experts_and_seeded():
    t = synth.hash_table(300, 16, 6, seed=3)
    assert t.shape == (300, 6) and t.dtype == np.int32
    assert np.all((t >= 0) & (t < 16))
    assert all(len(set(r)) == 6 for r in t.tolist())
    np.testing.assert_array_equal(t, synth.hash_table(300, 16, 6, seed=3))
    assert not np.array_equal(t, synth.hash_table(300, 16, 6, seed=4))
    # every expert shows up in about the same share of rows
    counts = np.bincount(t.ravel(), minlength=16)
    assert counts.min() > 0.7 * counts.mean() and counts.max() < 1.3 * counts.mean()
    ids = synth.token_ids(1000, 300, seed=3)
    assert ids.dtype == np.int32 and ids.min() >= 0 and ids.max() < 300
