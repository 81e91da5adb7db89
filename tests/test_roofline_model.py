"""The byte/FLOP model used for roofline fractions, pinned to the closed forms the pages print."""
import math

import pytest

from conftest import golden_kv
from routed_expert_ffn_moe_gb300 import roofline as R

G = golden_kv("closed_forms.txt")


def f(key):
    return float(G[key])


def test_v3_expert_params():
    assert R.expert_params(7168, 2048) == int(G["v3_expert_params"])


def test_v4pro_expert_params_and_flops():
    assert R.expert_params(7168, 3072) / 1e6 == pytest.approx(f("v4pro_expert_params_M"), abs=0.005)
    assert R.pair_flops(7168, 3072) / 1e6 == pytest.approx(f("v4pro_pair_MFLOPs"), abs=0.005)
    assert 7 * R.pair_flops(7168, 3072) / 1e6 == pytest.approx(f("v4pro_token_layer_MFLOPs"), abs=0.01)


def test_qwen3_layer_t1():
    h, ff, k = 4096, 1536, 8
    bytes_ = k * R.expert_bytes(h, ff, "bf16")
    assert R.mib(bytes_) == f("qwen3_layer_T1_MiB")
    assert R.mib(R.expert_bytes(h, ff, "bf16")) == f("qwen3_expert_MiB")
    flops = k * R.pair_flops(h, ff)
    assert flops == pytest.approx(f("qwen3_layer_T1_FLOPs"), rel=0.005)
    assert bytes_ / 3350e9 * 1e6 == pytest.approx(f("qwen3_layer_T1_us_at_3350GBps"), abs=0.05)
    assert flops / 989.4e12 * 1e6 == pytest.approx(f("qwen3_layer_T1_us_at_989TFLOPs"), abs=0.005)
    # eq. 6-2: the T=1 layer is bandwidth-bound, MFU <= 0.31 / 90.1 ~ 0.3 %
    t = R.roofline_time(flops, bytes_, 989.4e12, 3350e9)
    assert t == bytes_ / 3350e9 and (flops / 989.4e12) / t == pytest.approx(0.0034, abs=0.0002)


def test_qwen3_prefill_8192():
    h, ff, E, k, T = 4096, 1536, 128, 8, 8192
    all_bytes = E * R.expert_bytes(h, ff, "bf16")
    assert R.gib(all_bytes) == f("qwen3_all_experts_GiB")
    flops = T * k * R.pair_flops(h, ff)
    assert flops / 1e12 == pytest.approx(f("qwen3_T8192_TFLOPs"), abs=0.005)
    assert all_bytes / 3350e9 * 1e3 == pytest.approx(f("qwen3_T8192_ms_hbm"), abs=0.005)
    assert flops / 989.4e12 * 1e3 == pytest.approx(f("qwen3_T8192_ms_compute"), abs=0.005)
    assert R.roofline_time(flops, all_bytes, 989.4e12, 3350e9) == flops / 989.4e12


def test_eq_6_8_and_batch_reuse():
    act = R.expected_active(128, 8, 8)
    assert round(act) == int(G["eq68_E128_k8_m8_active"])
    assert R.gib(act * R.expert_bytes(4096, 1536, "bf16")) == pytest.approx(
        f("eq68_E128_k8_m8_GiB"), abs=0.05)
    assert R.mib(8 * R.expert_bytes(4096, 1536, "bf16")) == f("concentrated_64tok_MiB")
    # limits: one token hits exactly k experts; huge batches hit all of them
    assert R.expected_active(256, 8, 1) == pytest.approx(8.0)
    assert R.expected_active(256, 8, 10 ** 6) == pytest.approx(256.0)


@pytest.mark.parametrize("B", [16, 32, 64, 128, 256, 512])
def test_u_of_b_table(B):
    assert R.expected_active_u(384, 6, B) == pytest.approx(f(f"U_B{B}"), abs=0.006)


def test_fp8_expert_bytes_include_block_scales():
    d, ff = 7168, 2048
    assert R.expert_bytes(d, ff, "fp8") == 3 * d * ff + 4 * (3 * (d // 128) * (ff // 128))
    assert R.gate_up_bytes(d, ff, "fp8", 1) + R.down_bytes(d, ff, "fp8", 1) == R.expert_bytes(d, ff, "fp8")
    assert R.gate_up_bytes(d, ff, "bf16", 3) + R.down_bytes(d, ff, "bf16", 3) == 3 * R.expert_bytes(d, ff, "bf16")


def test_layer_flops_formula():
    # V3 decode T=256: 2*T*(k+1)*3*d*f + 2*T*d*E
    T, d, E, k, ff = 256, 7168, 256, 8, 2048
    assert R.layer_flops(T, d, E, k, ff, 1) == 2 * T * 9 * 3 * d * ff + 2 * T * d * E
    assert R.layer_flops(T, d, E, k, ff, 1) / 1e12 == pytest.approx(0.204, abs=0.001)
    assert not math.isnan(R.layer_bytes(T, d, E, ff, 1, "bf16", 255.9))


def test_fp4_expert_is_the_pages_33_mb_plus_its_scales():
    # "DeepSeek-V4-Pro on NVIDIA H200", 0.1.2 and 3.2: a routed expert of 3 x 7168 x 3072 =
    # 66.06M parameters takes about 33 MB in FP4; MXFP4 adds one scale byte per 32 elements
    d, ff = 7168, 3072
    params = R.expert_params(d, ff)
    assert params / 1e6 == pytest.approx(66.06, abs=0.01)
    elem = params // 2
    assert elem / 1e6 == pytest.approx(33.03, abs=0.01)
    assert R.expert_bytes(d, ff, "mxfp4") == elem + params // 32
    assert (R.gate_up_bytes(d, ff, "mxfp4", 2) + R.down_bytes(d, ff, "mxfp4", 2)
            == 2 * R.expert_bytes(d, ff, "mxfp4"))
