"""The oracle's pins catch plausible mistakes: each case plants one mistake in a copy of the
oracle's C source (a dropped term, a wrong sign, index, bias, order or operand), builds it, and
runs the pins (tests/test_oracle_pins.py) against that build in a subprocess; at least one pin
must fail. A copy without a planted mistake must pass them all. Every planted mistake keeps
every memory access in bounds, so a mutant can only compute wrong values."""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

MUTANTS = [
    # number formats
    ("bf16_shift", "(uint32_t)h << 16", "(uint32_t)h << 15"),
    ("e4m3_exponent_bias", "ldexp(1.0 + (double)m / 8.0, E - 7)",
     "ldexp(1.0 + (double)m / 8.0, E - 8)"),
    ("e4m3_subnormal_scale", "ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    ("e2m1_exponent_bias", "ldexp(1.0 + 0.5 * m, E - 1)", "ldexp(1.0 + 0.5 * m, E)"),
    ("e8m0_bias", "ldexp(1.0, (int)e - 127)", "ldexp(1.0, (int)e - 128)"),
    ("fp8_scale_row_stride_dropped", "(r / 128) * (cols / 128) + (c / 128)",
     "(r / 128) + (c / 128)"),
    ("mxfp4_nibble_order", "(c & 1) ? pair >> 4 : pair & 15", "(c & 1) ? pair & 15 : pair >> 4"),
    ("mxfp4_scale_block_width", "r * (cols / 32) + c / 32", "r * (cols / 32) + c / 64"),
    # router
    ("router_butterfly_reversed", "for (int off = 16; off >= 1; off /= 2)",
     "for (int off = 1; off <= 16; off *= 2)"),
    ("router_bias_sign", "lane[0] + bias[e]", "lane[0] - bias[e]"),
    ("topk_ascending", "if (p->l > q->l) return -1;\n  if (p->l < q->l) return 1;",
     "if (p->l > q->l) return 1;\n  if (p->l < q->l) return -1;"),
    ("topk_ties_to_higher_index", "return (p->e > q->e) - (p->e < q->e);",
     "return (p->e < q->e) - (p->e > q->e);"),
    ("gate_not_renormalised", "const double g = p[order[j].e] / zsel;",
     "const double g = p[order[j].e];"),
    ("hash_gate_not_renormalised", "const double g = exp((double)l[row[j]] - lmax) / z / zsel;",
     "const double g = exp((double)l[row[j]] - lmax) / z;"),
    # permutation
    ("permute_tokens_descending",
     "for (int t = 0; t < T; ++t)\n    for (int j = 0; j < k; ++j) {\n      const int e = topk_idx",
     "for (int t = T - 1; t >= 0; --t)\n    for (int j = 0; j < k; ++j) {\n      const int e = topk_idx"),
    ("shared_segment_end_missing", "offsets[E + 1] = (int32_t)(run + (int64_t)n_shared * T);",
     "offsets[E + 1] = (int32_t)(run);"),
    # expert FFN
    ("matvec_columns_reversed", "weight(wdtype, w, s, cols, row0 + r, c) * x[c]",
     "weight(wdtype, w, s, cols, row0 + r, cols - 1 - c) * x[c]"),
    ("gate_reads_up_rows", "oracle_matvec(wdtype, w13, s13, d, 0, f, xv, g);",
     "oracle_matvec(wdtype, w13, s13, d, f, f, xv, g);"),
    ("up_reads_gate_rows", "oracle_matvec(wdtype, w13, s13, d, f, f, xv, u);",
     "oracle_matvec(wdtype, w13, s13, d, 0, f, xv, u);"),
    ("silu_sign", "g[r] / (1.0 + exp(-g[r]))", "g[r] / (1.0 + exp(g[r]))"),
    ("silu_dropped", "g[r] = silu * u[r];", "g[r] = g[r] * u[r];"),
    # combine and the layer
    ("shared_output_dropped", "if (n_shared)\n      for (int c = 0; c < d; ++c) out[c] += y_perm",
     "if (0)\n      for (int c = 0; c < d; ++c) out[c] += y_perm"),
    ("combine_shared_row_fixed", "y_perm[((int64_t)T * k + t) * d + c]",
     "y_perm[((int64_t)T * k) * d + c]"),
    ("combine_gate_weight_dropped", "out[c] += g * row[c];", "out[c] += row[c];"),
    ("layer_segment_lookup_off_by_one", "while (offsets[e + 1] <= slot) ++e;",
     "while (offsets[e + 1] < slot) ++e;"),
]


def run_pins(tmp_path, source: str) -> subprocess.CompletedProcess:
    src = tmp_path / "moe_oracle.c"
    src.write_text(source)
    lib = oracle.compile_source(str(src), str(tmp_path / "libmoe_oracle.so"))
    env = dict(os.environ, MOE_ORACLE_LIB=lib)
    return subprocess.run(
        [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
         "-x", "-q", "-p", "no:cacheprovider"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_unmodified_copy_passes_the_pins(tmp_path):
    r = run_pins(tmp_path, open(SRC).read())
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(tmp_path, name, old, new):
    source = open(SRC).read()
    assert source.count(old) == 1, f"{name}: the planted line must occur exactly once"
    r = run_pins(tmp_path, source.replace(old, new))
    assert r.returncode == 1, f"{name} survived the pins:\n{r.stdout[-2000:]}"


# Mistakes planted in oracle.token_outputs (the per-token output the full-size GPU checks use):
# each mutated copy of the function replaces the original for the duration of the case, and the
# token_outputs pins must fail.
PY_MUTANTS = [
    ("token_outputs_gate_column_shifted", "y[i] += topk_w64[i, j] * yr",
     "y[i] += topk_w64[i, (j + 1) % topk_w64.shape[1]] * yr"),
    ("token_outputs_rows_paired_in_reverse", "for (i, j), yr in zip(pairs, ye):",
     "for (i, j), yr in zip(pairs, ye[::-1]):"),
    ("token_outputs_shared_dropped", "if shared is not None:", "if False:"),
    ("token_outputs_shared_twice",
     "y += expert_rows(x_rows, shared.w13, shared.w2, wdtype, shared.s13, shared.s2)",
     "y += 2 * expert_rows(x_rows, shared.w13, shared.w2, wdtype, shared.s13, shared.s2)"),
    ("token_outputs_expert_of_wrong_choice", "by_expert.setdefault(int(e), []).append((i, j))",
     "by_expert.setdefault(int(topk_idx[i][0]), []).append((i, j))"),
]


def _run_token_output_pins():
    import test_oracle_pins as pins
    for name, over in pins.TOKEN_OUTPUT_CASES:
        pins.test_token_outputs_equal_the_whole_layer(name, over)
    for wd in ("bf16", "fp8"):
        pins.test_token_outputs_of_hash_routing_equal_the_dense_masked_evaluation(wd)


def test_unmodified_token_outputs_passes_its_pins():
    _run_token_output_pins()


@pytest.mark.parametrize("name,old,new", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_planted_mistake_in_token_outputs_fails_a_pin(monkeypatch, name, old, new):
    import inspect
    src = inspect.getsource(oracle.token_outputs)
    assert src.count(old) == 1, f"{name}: the planted line must occur exactly once"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), f"<{name}>", "exec"), ns)
    monkeypatch.setattr(oracle, "token_outputs", ns["token_outputs"])
    with pytest.raises(AssertionError):
        _run_token_output_pins()
