"""Why the FP8 weights run as W8A16 and not W8A8: the arithmetic of the W8A8 variant, emulated.

The CANN page runs V4's experts with 8-bit activations (W8A8 on A3, MXFP8 on 950;
"CANN DeepSeek-V4推理优化", 量化策略), and DeepSeek's FP8 GEMMs saturate the tensor cores from
m > 4096 ("DeepSeek V3/R1 Inference Efficiency (1)", section 2), so an FP8 x FP8 MMA would double
the tensor rate of large batches. Its activations would be E4M3 codes with one fp32 scale per
token and 128-wide K block (scale = block amax / 448, codes by round-to-nearest-even). E4M3 keeps
3 fraction bits, so each activation carries up to 2^-4 relative error, and the layer output
inherits it: this test computes the layer output of that arithmetic on the V3 shape with FP8
block-scaled weights (the token-batch sweep's weights, first tokens of its batch, three experts
with Dirichlet gate weights) in fp64, and its relative L2 distance from the exact layer. It is
above the 3e-2 acceptance bar of FP8 weights, whether h is quantised too (W8A8 in both GEMMs) or
x alone (gate/up only), so the W8A8 variant is not built. A GPU kernel would reproduce these
figures up to fp32 accumulation order, which is far smaller."""
import numpy as np
import pytest

import oracle
import synth

BAR = 3e-2


def _e4m3_table():
    v = np.array([oracle.e4m3_value(c) for c in range(256)])
    v[np.isnan(v)] = 0.0
    return v


def _dequant(table, ew, which):
    q, s = getattr(ew, which), getattr(ew, "s" + which[1:])
    return table[q] * np.kron(s.astype(np.float64), np.ones((128, 128)))


def _quant_rows_e4m3(table, a, blk=128):
    """Per row and 128-wide column block: s = amax / 448 (1 if amax = 0), codes by RNE
    (synth's E4M3 encoder), value = code * s."""
    out = np.empty_like(a)
    for b in range(0, a.shape[1], blk):
        v = a[:, b:b + blk]
        amax = np.abs(v).max(axis=1, keepdims=True)
        s = np.where(amax > 0, amax / 448.0, 1.0)
        out[:, b:b + blk] = table[synth.f32_to_e4m3((v / s).astype(np.float32))] * s
    return out


@pytest.mark.timeout(600)
def test_w8a8_layer_error_is_above_the_fp8_bar():
    cfg = synth.get_config("sweep_fp8_T4096")
    table = _e4m3_table()
    ntok, nexp = 4, 3
    x = oracle.bf16_to_f64(synth.host_x(cfg, tokens=range(ntok)))
    xq = _quant_rows_e4m3(table, x)
    g = np.random.default_rng(0).dirichlet(np.ones(nexp), size=ntok)
    y_exact = y_w8a8 = y_x_only = 0.0
    for j in range(nexp):
        ew = synth.host_expert(cfg, j)
        W13, Wd = _dequant(table, ew, "w13"), _dequant(table, ew, "w2")

        def ffn(xx, quant_h):
            G, U = xx @ W13[: cfg.f].T, xx @ W13[cfg.f:].T
            h = G / (1.0 + np.exp(-G)) * U
            return (_quant_rows_e4m3(table, h) if quant_h else h) @ Wd.T

        y_exact = y_exact + g[:, j:j + 1] * ffn(x, False)
        y_w8a8 = y_w8a8 + g[:, j:j + 1] * ffn(xq, True)
        y_x_only = y_x_only + g[:, j:j + 1] * ffn(xq, False)
    rel = lambda y: float(np.linalg.norm(y - y_exact) / np.linalg.norm(y_exact))  # noqa: E731
    r_both, r_x = rel(y_w8a8), rel(y_x_only)
    print(f"W8A8 layer rel-L2: {r_both:.4f} (x and h in E4M3), {r_x:.4f} (x alone)")
    assert r_both > BAR and r_x > BAR
