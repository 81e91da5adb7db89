"""Byte and FLOP model of the MoE layer, and the roofline it is measured against.

Closed forms from the pages:
  * one expert = three matrices of h x d_ff parameters; one token-expert pair costs 6*h*d_ff
    FLOPs ("DeepSeek-V4-Pro on NVIDIA H200", 3.2; "DeepSeek V3/R1 Inference Efficiency (1)",
    Parameters: 7168 x 2048 x 3 = 44M per expert);
  * expected distinct experts hit by m tokens choosing k of E each, uniformly and independently:
    E[1 - (1 - k/E)^m] ("第 6 章 超節點", 6.3.2, eq. 6-8); the H200 report's variant
    U(B) = E(1 - (1 - 1/E)^(kB)) ("DeepSeek-V4-Pro on NVIDIA H200", 3.2 and the section 6 table);
  * T_op = max(F/P, V/B_HBM) ("第 6 章 超節點", 6.1.2, eq. 6-2).

Algorithmic bytes of one layer = weights (and block scales) of every expert that received at
least one token + the shared expert + W_g + x + y. Intermediates (gathered x, h, per-slot expert
outputs) are implementation traffic and are not counted.
"""
from __future__ import annotations


def expert_params(d: int, f: int) -> int:
    """Parameters of one SwiGLU expert: gate, up ([f, d] each) and down ([d, f])."""
    return 3 * d * f


def pair_flops(d: int, f: int) -> int:
    """FLOPs of one token through one expert (three GEMVs, 2 FLOPs per multiply-add)."""
    return 6 * d * f


def expected_active(E: int, k: int, m: int) -> float:
    """Eq. 6-8: expected number of distinct experts hit by a batch of m tokens."""
    return E * (1.0 - (1.0 - k / E) ** m)


def expected_active_u(E: int, k: int, B: int) -> float:
    """The H200 report's U(B) = E (1 - (1 - 1/E)^(k B))."""
    return E * (1.0 - (1.0 - 1.0 / E) ** (k * B))


def matrix_bytes(rows: int, cols: int, wdtype: str) -> int:
    """HBM bytes of one [rows, cols] weight matrix with its scales: bf16 (2 bytes an element);
    E4M3 (1 byte) plus one fp32 scale per 128x128 block; MXFP4 (half a byte) plus one E8M0
    byte per 32 elements."""
    n = rows * cols
    if wdtype == "bf16":
        return 2 * n
    if wdtype == "fp8":
        return n + 4 * (rows // 128) * (cols // 128)
    return n // 2 + n // 32


def expert_bytes(d: int, f: int, wdtype: str) -> int:
    """HBM bytes of one expert's weights (gate, up, down) with their scales."""
    return matrix_bytes(2 * f, d, wdtype) + matrix_bytes(d, f, wdtype)


def layer_bytes(T: int, d: int, E: int, f: int, n_shared: int, wdtype: str,
                n_active: float) -> float:
    """Algorithmic bytes of one layer with n_active routed experts hit."""
    return ((n_active + n_shared) * expert_bytes(d, f, wdtype)
            + E * d * 2          # router weight W_g, bf16
            + T * d * 2          # x, bf16
            + T * d * 2)         # y, bf16


def layer_flops(T: int, d: int, E: int, k: int, f: int, n_shared: int) -> int:
    """Expert FLOPs of T tokens through k routed + n_shared experts, plus the router GEMM."""
    return T * (k + n_shared) * pair_flops(d, f) + 2 * T * d * E


def roofline_time(flops: float, bytes_: float, peak_flops: float, peak_bw: float) -> float:
    """Eq. 6-2: lower bound on the time of an operator that overlaps compute and memory."""
    return max(flops / peak_flops, bytes_ / peak_bw)


def gate_up_bytes(d: int, f: int, wdtype: str, n_experts_run: int) -> int:
    """Algorithmic bytes of the gate/up phase: the gate and up weights (+ scales) of every expert
    that runs (routed experts hit + shared)."""
    return n_experts_run * matrix_bytes(2 * f, d, wdtype)


def down_bytes(d: int, f: int, wdtype: str, n_experts_run: int) -> int:
    return n_experts_run * matrix_bytes(d, f, wdtype)


def mib(x: float) -> float:
    return x / 2 ** 20


def gib(x: float) -> float:
    return x / 2 ** 30

