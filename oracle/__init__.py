"""CPU oracle for the routed-expert MoE FFN layer -- TEST INFRASTRUCTURE ONLY.

Thin numpy/ctypes wrapper over moe_oracle.c (plain C, fp64 except the fp32 router logits that
decide the top-k choice). Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg
use it. It imports nothing from the CUDA library, and the CUDA library imports nothing from it.

Parity pins: every function here is checked by tests/test_oracle_pins.py against the pages'
worked example and closed forms, library-routine reductions (numpy matmul / lexsort), brute
force on tiny inputs and invariants. No function is left unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
# MOE_ORACLE_LIB points the wrapper at another build of this interface: the mutation test loads
# builds with a planted mistake this way, to show that the pins catch each one.
_LIB = os.environ.get("MOE_ORACLE_LIB") or os.path.join(_HERE, "libmoe_oracle.so")

WD = {"bf16": 0, "fp8": 1, "mxfp4": 2}


def compile_source(src: str, out: str) -> str:
    """gcc -O2, no fp contraction (so results do not depend on the host's FMA units)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def build(force: bool = False) -> str:
    if os.environ.get("MOE_ORACLE_LIB"):  # another build, made by whoever set the variable
        return _LIB
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    return compile_source(_SRC, _LIB)


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        L.oracle_bf16_value.restype = ctypes.c_double
        L.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        L.oracle_e4m3_value.restype = ctypes.c_double
        L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        L.oracle_e2m1_value.restype = ctypes.c_double
        L.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
        L.oracle_e8m0_value.restype = ctypes.c_double
        L.oracle_e8m0_value.argtypes = [ctypes.c_uint8]
        L.oracle_router_logits.argtypes = [vp, vp, vp, i32, i32, i32, vp]
        L.oracle_route.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        L.oracle_permute.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp]
        L.oracle_route_hash.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, vp]
        L.oracle_matvec.argtypes = [i32, vp, vp, i64, i64, i64, vp, vp]
        L.oracle_expert_rows.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.oracle_combine.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp]
        L.oracle_moe_layer.argtypes = [i32] * 7 + [vp] * 16
        for fn in ("oracle_router_logits", "oracle_route", "oracle_route_hash", "oracle_permute",
                   "oracle_matvec",
                   "oracle_expert_rows", "oracle_combine", "oracle_moe_layer"):
            getattr(L, fn).restype = None
        _lib = L
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ---- formats -------------------------------------------------------------------------------

def bf16_value(h: int) -> float:
    return lib().oracle_bf16_value(int(h))


def e4m3_value(q: int) -> float:
    return lib().oracle_e4m3_value(int(q))


def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(int(code))


def e8m0_value(e: int) -> float:
    return lib().oracle_e8m0_value(int(e))


def _scales(s, wdtype):
    """Scales as the C side reads them: fp32 for FP8, E8M0 bytes for MXFP4."""
    return _c(s, np.uint8 if wdtype == "mxfp4" else np.float32)


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    """Array of bf16 bit patterns -> fp64 values (the upper half of an fp32)."""
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---- a1 ------------------------------------------------------------------------------------

def router_logits(x, wg, bias=None):
    x, wg = _c(x, np.uint16), _c(wg, np.uint16)
    bias = _c(bias, np.float32)
    T, d = x.shape
    E = wg.shape[0]
    assert d % 8 == 0
    out = np.empty((T, E), dtype=np.float32)
    lib().oracle_router_logits(_p(x), _p(wg), _p(bias), T, d, E, _p(out))
    return out


def route(logits, k):
    """-> topk_idx int32 [T,k], topk_w float32 [T,k], topk_w64 float64 [T,k]."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    w64 = np.empty((T, k), np.float64)
    lib().oracle_route(_p(logits), T, E, k, _p(idx), _p(w), _p(w64))
    return idx, w, w64


def route_hash(logits, token_ids, tid2eid):
    """Hash routing: the k experts of each token from tid2eid[token_id] (table order) and the
    soft router's renormalised gate at them. -> topk_idx, topk_w (fp32), topk_w64."""
    logits = _c(logits, np.float32)
    tid = _c(token_ids, np.int32)
    table = _c(tid2eid, np.int32)
    T, E = logits.shape
    k = table.shape[1]
    assert tid.shape == (T,) and np.all((tid >= 0) & (tid < table.shape[0]))
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    w64 = np.empty((T, k), np.float64)
    lib().oracle_route_hash(_p(logits), _p(tid), _p(table), T, E, k, _p(idx), _p(w), _p(w64))
    return idx, w, w64


# ---- a2 ------------------------------------------------------------------------------------

def permute(topk_idx, E, n_shared=1):
    """-> expert_offsets int32 [E+2], perm_token int32 [T*k], inv_slot int32 [T*k]."""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    off = np.empty(E + 2, np.int32)
    perm = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    lib().oracle_permute(_p(idx), T, E, k, n_shared, _p(off), _p(perm), _p(inv))
    return off, perm, inv


# ---- a3 + a4 -------------------------------------------------------------------------------

def matvec(w, x, wdtype="bf16", s=None, row0=0, nrows=None):
    """y[r] = sum_c W[row0 + r][c] x[c] in fp64, W row-major bf16 bits, E4M3 codes, or MXFP4
    code pairs ([rows, cols/2] bytes)."""
    w = _c(w, np.uint16 if wdtype == "bf16" else np.uint8)
    x = _c(x, np.float64)
    rows, cols = w.shape
    if wdtype == "mxfp4":
        cols *= 2
    nrows = rows - row0 if nrows is None else nrows
    y = np.empty(nrows, np.float64)
    lib().oracle_matvec(WD[wdtype], _p(w), _p(_scales(s, wdtype)), cols, row0, nrows, _p(x), _p(y))
    return y


def expert_rows(xrows, w13, w2, wdtype="bf16", s13=None, s2=None, want_h=False):
    """SwiGLU expert on rows xrows [n, d] (bf16 bits): returns y [n, d] fp64 (and h [n, f])."""
    xrows = _c(xrows, np.uint16)
    n, d = xrows.shape
    wt = np.uint16 if wdtype == "bf16" else np.uint8
    w13, w2 = _c(w13, wt), _c(w2, wt)
    f = w13.shape[0] // 2
    per_byte = 2 if wdtype == "mxfp4" else 1
    assert w13.shape == (2 * f, d // per_byte) and w2.shape == (d, f // per_byte)
    y = np.empty((n, d), np.float64)
    h = np.empty((n, f), np.float64) if want_h else None
    lib().oracle_expert_rows(_p(xrows), n, d, f, WD[wdtype], _p(w13), _p(_scales(s13, wdtype)),
                             _p(w2), _p(_scales(s2, wdtype)), _p(y), _p(h))
    return (y, h) if want_h else y


# ---- a5 ------------------------------------------------------------------------------------

def combine(y_perm, inv_slot, topk_w, T, k, n_shared=1):
    y_perm = _c(y_perm, np.float64)
    d = y_perm.shape[1]
    y = np.empty((T, d), np.float64)
    lib().oracle_combine(_p(y_perm), _p(_c(inv_slot, np.int32)), _p(_c(topk_w, np.float64)), T, k,
                         d, n_shared, _p(y))
    return y


# ---- whole layer ---------------------------------------------------------------------------

def moe_layer(cfg, inputs):
    """Every output of the layer for a (small) config; inputs from synth.host_inputs."""
    T, d, E, k, f, S = cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.n_shared
    ex = inputs.experts
    w13 = np.ascontiguousarray(np.stack([e.w13 for e in ex]))
    w2 = np.ascontiguousarray(np.stack([e.w2 for e in ex]))
    scaled = cfg.wdtype in ("fp8", "mxfp4")
    s13 = _scales(np.stack([e.s13 for e in ex]), cfg.wdtype) if scaled else None
    s2 = _scales(np.stack([e.s2 for e in ex]), cfg.wdtype) if scaled else None
    slots = T * k + S * T
    out = dict(logits=np.empty((T, E), np.float32), topk_idx=np.empty((T, k), np.int32),
               topk_w=np.empty((T, k), np.float32), topk_w64=np.empty((T, k), np.float64),
               expert_offsets=np.empty(E + 2, np.int32), perm_token=np.empty(T * k, np.int32),
               inv_slot=np.empty(T * k, np.int32), y_perm=np.empty((slots, d), np.float64),
               y=np.empty((T, d), np.float64))
    x = _c(inputs.x, np.uint16)
    wg = _c(inputs.wg, np.uint16)
    bias = _c(inputs.bias, np.float32)
    lib().oracle_moe_layer(T, d, E, k, f, S, WD[cfg.wdtype], _p(x), _p(wg), _p(bias), _p(w13),
                           _p(s13), _p(w2), _p(s2), _p(out["logits"]), _p(out["topk_idx"]),
                           _p(out["topk_w"]), _p(out["topk_w64"]), _p(out["expert_offsets"]),
                           _p(out["perm_token"]), _p(out["inv_slot"]), _p(out["y_perm"]),
                           _p(out["y"]))
    return out


def token_outputs(x_rows, topk_idx, topk_w64, experts: dict, shared, wdtype="bf16"):
    """y for a sample of tokens, straight from the definition (tokens are independent):
    y_t = shared(x_t) + sum_j g_tj * expert_{e_tj}(x_t). `experts` maps expert id ->
    synth.ExpertWeights; `shared` is the shared expert's weights or None."""
    x_rows = _c(x_rows, np.uint16)
    n, d = x_rows.shape
    y = np.zeros((n, d), np.float64)
    if shared is not None:
        y += expert_rows(x_rows, shared.w13, shared.w2, wdtype, shared.s13, shared.s2)
    by_expert = {}
    for i in range(n):
        for j, e in enumerate(topk_idx[i]):
            by_expert.setdefault(int(e), []).append((i, j))
    for e, pairs in sorted(by_expert.items()):
        rows = np.array([i for i, _ in pairs])
        ew = experts[e]
        ye = expert_rows(x_rows[rows], ew.w13, ew.w2, wdtype, ew.s13, ew.s2)
        for (i, j), yr in zip(pairs, ye):
            y[i] += topk_w64[i, j] * yr
    return y
