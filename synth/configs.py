"""The workloads: shapes, weight format and router kind of each synthetic MoE layer.

Shapes follow the pages: DeepSeek-V3 (d=7168, 256 routed + 1 shared experts, top-8, expert
intermediate 2048; "DeepSeek V3/R1 Inference Efficiency (1)", Parameters) and DeepSeek-V4-Pro
(d=7168, 384 routed + 1 shared, top-6, intermediate 3072; "DeepSeek-V4-Pro on NVIDIA H200",
section 2.1).
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class MoeConfig:
    name: str
    T: int          # tokens in the batch
    d: int          # hidden size
    E: int          # routed experts
    k: int          # routed experts chosen per token
    f: int          # expert intermediate size
    n_shared: int   # always-on shared experts (0 or 1)
    wdtype: str     # "bf16", "fp8" (E4M3 with fp32 scales per 128x128 block) or "mxfp4"
                    # (E2M1 with E8M0 scales per 32 consecutive elements of a row)
    router: str     # "uniform" (plain logits) or "zipf" (logits + Zipf popularity bias)
    seed: int = 0

    @property
    def n_experts(self) -> int:
        return self.E + self.n_shared

    @property
    def slots(self) -> int:
        """Rows of the permuted expert input/output: T*k routed + T*n_shared shared."""
        return self.T * self.k + self.T * self.n_shared


CONFIGS = {
    "tiny": MoeConfig("tiny", T=16, d=256, E=8, k=2, f=128, n_shared=1, wdtype="bf16",
                      router="uniform"),
    "v3_decode": MoeConfig("v3_decode", T=256, d=7168, E=256, k=8, f=2048, n_shared=1,
                           wdtype="bf16", router="uniform"),
    "v4pro_decode": MoeConfig("v4pro_decode", T=32, d=7168, E=384, k=6, f=3072, n_shared=1,
                              wdtype="fp8", router="uniform"),
    # V4-Pro's routed experts in FP4, the format its public description gives them
    # ("DeepSeek-V4-Pro on NVIDIA H200", 0.1.3; "CANN DeepSeek-V4推理优化", 量化策略: MXFP4)
    "v4pro_decode_fp4": MoeConfig("v4pro_decode_fp4", T=32, d=7168, E=384, k=6, f=3072,
                                  n_shared=1, wdtype="mxfp4", router="uniform"),
    "skewed_prefill": MoeConfig("skewed_prefill", T=4096, d=7168, E=256, k=8, f=2048,
                                n_shared=1, wdtype="bf16", router="zipf"),
}

SWEEP_T = (1, 8, 64, 256, 1024, 4096, 16384)


def sweep_config(T: int) -> MoeConfig:
    """V3 shape with FP8 block-scaled expert weights and a plain router, at token batch T."""
    return MoeConfig(f"sweep_fp8_T{T}", T=T, d=7168, E=256, k=8, f=2048, n_shared=1,
                     wdtype="fp8", router="uniform")


def sweep_fp4_config(T: int) -> MoeConfig:
    """V3 shape with MXFP4 expert weights and a plain router, at token batch T."""
    return MoeConfig(f"sweep_fp4_T{T}", T=T, d=7168, E=256, k=8, f=2048, n_shared=1,
                     wdtype="mxfp4", router="uniform")


def get_config(name: str, **overrides) -> MoeConfig:
    if name.startswith("sweep_fp8_T"):
        cfg = sweep_config(int(name[len("sweep_fp8_T"):]))
    elif name.startswith("sweep_fp4_T"):
        cfg = sweep_fp4_config(int(name[len("sweep_fp4_T"):]))
    else:
        cfg = CONFIGS[name]
    return replace(cfg, **overrides) if overrides else cfg
