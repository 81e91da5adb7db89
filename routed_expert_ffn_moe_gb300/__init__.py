"""Python binding of the GB300 routed-expert MoE FFN library (include/moe.h).

Argument marshalling only: every step of the layer runs in the CUDA kernels of
libmoe_gb300.so. Tensors are torch CUDA tensors (PyTorch provides device memory and streams);
the functions below pass their device pointers to the C ABI. There is no CPU fallback: if the
library is missing or was not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os

__all__ = ["MoeError", "MoeShape", "MOE_W_BF16", "MOE_W_FP8_E4M3_B128", "MOE_W_MXFP4_E8M0_B32",
           "load", "lib_path",
           "moe_workspace_size", "moe_route", "moe_route_hash", "moe_route_noalloc", "moe_permute",
           "moe_expert_ffn", "moe_combine", "moe_forward",
           "moe_check_device_status", "moe_selftest_bounded_wait", "moe_profile_enable",
           "moe_profile_read",
           "moe_last_error_string", "shape_of", "MoeLayer", "EXPORTED"]

MOE_W_BF16, MOE_W_FP8_E4M3_B128, MOE_W_MXFP4_E8M0_B32 = 0, 1, 2
WDTYPES = {"bf16": MOE_W_BF16, "fp8": MOE_W_FP8_E4M3_B128, "mxfp4": MOE_W_MXFP4_E8M0_B32}
STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED",
          -3: "MOE_ERR_WORKSPACE", -4: "MOE_ERR_CUDA", -5: "MOE_ERR_DEVICE_TIMEOUT",
          -6: "MOE_ERR_DEVICE_BOUNDS"}
EXPORTED = ("moe_workspace_size", "moe_route", "moe_route_hash", "moe_route_noalloc", "moe_permute",
            "moe_expert_ffn",
            "moe_combine", "moe_forward",
            "moe_check_device_status", "moe_selftest_bounded_wait", "moe_profile_enable",
            "moe_profile_read", "moe_last_error_string")

_PKG = os.path.dirname(os.path.abspath(__file__))


def lib_path() -> str:
    return os.path.join(_PKG, "libmoe_gb300.so")


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}: {msg}")
        self.status = status


class MoeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("f", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("wdtype", ctypes.c_int32)]


_lib = None


def load():
    """Loads libmoe_gb300.so. Raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it first "
                          "(python -m routed_expert_ffn_moe_gb300.build or __graft_entry__.build())")
    L = ctypes.CDLL(path)
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    shp = ctypes.POINTER(MoeShape)
    L.moe_workspace_size.restype = sz
    L.moe_workspace_size.argtypes = [shp]
    L.moe_route.restype = i32
    L.moe_route.argtypes = [shp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_route_hash.restype = i32
    L.moe_route_hash.argtypes = [shp, vp, vp, vp, vp, vp, ctypes.c_int32, vp, vp, vp, sz, vp]
    L.moe_route_noalloc.restype = i32
    L.moe_route_noalloc.argtypes = [shp, vp, vp, vp, vp, vp, vp]
    L.moe_permute.restype = i32
    L.moe_permute.argtypes = [shp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_expert_ffn.restype = i32
    L.moe_expert_ffn.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_combine.restype = i32
    L.moe_combine.argtypes = [shp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_forward.restype = i32
    L.moe_forward.argtypes = [shp] + [vp] * 15 + [sz, vp]
    L.moe_check_device_status.restype = i32
    L.moe_check_device_status.argtypes = [vp, vp]
    L.moe_selftest_bounded_wait.restype = i32
    L.moe_selftest_bounded_wait.argtypes = [vp, ctypes.c_uint32, vp]
    L.moe_profile_enable.restype = i32
    L.moe_profile_enable.argtypes = [i32]
    L.moe_profile_read.restype = i32
    L.moe_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                                   ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]
    L.moe_last_error_string.restype = ctypes.c_char_p
    L.moe_last_error_string.argtypes = []
    _lib = L
    return L


def _ptr(t):
    """Device pointer of a torch tensor (or an int address, or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str):
    if rc != 0:
        raise MoeError(rc, where, load().moe_last_error_string().decode(errors="replace"))


def shape_of(T, d, E, k, f, n_shared=1, wdtype=MOE_W_BF16) -> MoeShape:
    if isinstance(wdtype, str):
        wdtype = WDTYPES[wdtype]
    return MoeShape(T, d, E, k, f, n_shared, wdtype)


def moe_last_error_string() -> str:
    return load().moe_last_error_string().decode(errors="replace")


def moe_workspace_size(shape: MoeShape) -> int:
    return int(load().moe_workspace_size(ctypes.byref(shape)))


def _ws(ws):
    return _ptr(ws), (ws.numel() * ws.element_size() if hasattr(ws, "numel") else 0)


def moe_route(shape, x, wg, bias, topk_idx, topk_w, ws, stream=None, ws_bytes=None):
    wp, wb = _ws(ws)
    _check(load().moe_route(ctypes.byref(shape), _ptr(x), _ptr(wg), _ptr(bias), _ptr(topk_idx),
                            _ptr(topk_w), wp, wb if ws_bytes is None else ws_bytes,
                            _stream(stream)), "moe_route")


def moe_route_hash(shape, x, wg, bias, token_ids, tid2eid, topk_idx, topk_w, ws, stream=None,
                   ws_bytes=None):
    """Hash routing: experts from tid2eid [vocab, k] by token id, the soft router's gate."""
    wp, wb = _ws(ws)
    _check(load().moe_route_hash(ctypes.byref(shape), _ptr(x), _ptr(wg), _ptr(bias),
                                 _ptr(token_ids), _ptr(tid2eid), int(tid2eid.shape[0]),
                                 _ptr(topk_idx), _ptr(topk_w), wp,
                                 wb if ws_bytes is None else ws_bytes, _stream(stream)),
           "moe_route_hash")


def moe_route_noalloc(shape, x, wg, bias, topk_idx, topk_w, stream=None):
    """moe_route without a workspace (for callers that cannot allocate device memory): the
    library keeps the logits in a fixed 4 MiB device array, so T*E must be <= 2^20."""
    _check(load().moe_route_noalloc(ctypes.byref(shape), _ptr(x), _ptr(wg), _ptr(bias),
                                    _ptr(topk_idx), _ptr(topk_w), _stream(stream)),
           "moe_route_noalloc")


def moe_permute(shape, topk_idx, expert_offsets, perm_token, inv_slot, ws, stream=None,
                ws_bytes=None):
    wp, wb = _ws(ws)
    _check(load().moe_permute(ctypes.byref(shape), _ptr(topk_idx), _ptr(expert_offsets),
                              _ptr(perm_token), _ptr(inv_slot), wp,
                              wb if ws_bytes is None else ws_bytes, _stream(stream)), "moe_permute")


def moe_expert_ffn(shape, x, perm_token, expert_offsets, w13, s13, w2, s2, y_perm, ws,
                   stream=None, ws_bytes=None):
    wp, wb = _ws(ws)
    _check(load().moe_expert_ffn(ctypes.byref(shape), _ptr(x), _ptr(perm_token),
                                 _ptr(expert_offsets), _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2),
                                 _ptr(y_perm), wp, wb if ws_bytes is None else ws_bytes,
                                 _stream(stream)), "moe_expert_ffn")


def moe_combine(shape, y_perm, inv_slot, topk_w, y, ws, stream=None, ws_bytes=None):
    wp, wb = _ws(ws)
    _check(load().moe_combine(ctypes.byref(shape), _ptr(y_perm), _ptr(inv_slot), _ptr(topk_w),
                              _ptr(y), wp, wb if ws_bytes is None else ws_bytes, _stream(stream)),
           "moe_combine")


def moe_forward(shape, x, wg, bias, w13, s13, w2, s2, topk_idx, topk_w, expert_offsets,
                perm_token, inv_slot, y_perm, y, ws, stream=None, ws_bytes=None):
    """The four calls in one, with the shared expert's FFN overlapped with the routing."""
    wp, wb = _ws(ws)
    _check(load().moe_forward(ctypes.byref(shape), _ptr(x), _ptr(wg), _ptr(bias), _ptr(w13),
                              _ptr(s13), _ptr(w2), _ptr(s2), _ptr(topk_idx), _ptr(topk_w),
                              _ptr(expert_offsets), _ptr(perm_token), _ptr(inv_slot),
                              _ptr(y_perm), _ptr(y), wp, wb if ws_bytes is None else ws_bytes,
                              _stream(stream)), "moe_forward")


def moe_check_device_status(ws, stream=None):
    _check(load().moe_check_device_status(_ptr(ws), _stream(stream)), "moe_check_device_status")


def moe_selftest_bounded_wait(ws, limit_us, stream=None):
    """Launches a kernel whose wait never completes; after `limit_us` it records
    MOE_ERR_DEVICE_TIMEOUT in ws's status word (read it with moe_check_device_status)."""
    _check(load().moe_selftest_bounded_wait(_ptr(ws), int(limit_us), _stream(stream)),
           "moe_selftest_bounded_wait")


def moe_profile_enable(on: bool = True):
    _check(load().moe_profile_enable(1 if on else 0), "moe_profile_enable")


def moe_profile_read() -> dict:
    up, dn = ctypes.c_double(), ctypes.c_double()
    calls, launches = ctypes.c_int64(), ctypes.c_int64()
    _check(load().moe_profile_read(ctypes.byref(up), ctypes.byref(dn), ctypes.byref(calls),
                                   ctypes.byref(launches)), "moe_profile_read")
    return {"ms_gate_up": up.value, "ms_down": dn.value, "ffn_calls": calls.value,
            "kernel_launches": launches.value}


class MoeLayer:
    """The four calls chained on one stream with buffers allocated once (torch, on `device`).

    weights: dict with wg [E,d] bf16, bias [E] f32 or None, w13, w2 (bf16, uint8 E4M3 codes or
    uint8 MXFP4 code pairs), s13, s2 (fp32 block scales, uint8 E8M0 scales, or None). `forward(x)` returns y [T,d] bf16; intermediate tensors
    stay available as attributes (topk_idx, topk_w, expert_offsets, perm_token, inv_slot, y_perm).
    """

    def __init__(self, T, d, E, k, f, n_shared, wdtype, weights, device="cuda"):
        import torch
        self.shape = shape_of(T, d, E, k, f, n_shared, wdtype)
        self.w = weights
        dev = torch.device(device)
        slots = T * k + n_shared * T
        self.ws = torch.empty(max(moe_workspace_size(self.shape), 256), dtype=torch.uint8, device=dev)
        self.ws[:4].zero_()
        self.topk_idx = torch.empty(T, k, dtype=torch.int32, device=dev)
        self.topk_w = torch.empty(T, k, dtype=torch.float32, device=dev)
        self.expert_offsets = torch.empty(E + 2, dtype=torch.int32, device=dev)
        self.perm_token = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
        self.inv_slot = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
        self.y_perm = torch.empty(max(slots, 1), d, dtype=torch.float32, device=dev)
        self.y = torch.empty(T, d, dtype=torch.bfloat16, device=dev)

    def forward(self, x, stream=None):
        """The layer through moe_forward (one call; the shared expert overlaps the routing)."""
        w = self.w
        moe_forward(self.shape, x, w["wg"], w.get("bias"), w["w13"], w.get("s13"), w["w2"],
                    w.get("s2"), self.topk_idx, self.topk_w, self.expert_offsets, self.perm_token,
                    self.inv_slot, self.y_perm, self.y, self.ws, stream)
        return self.y

    def forward_hash(self, x, token_ids, tid2eid, stream=None):
        """The layer with hash routing (moe_route_hash, then permute, expert FFN, combine)."""
        w, s = self.w, self.shape
        moe_route_hash(s, x, w["wg"], w.get("bias"), token_ids, tid2eid, self.topk_idx,
                       self.topk_w, self.ws, stream)
        moe_permute(s, self.topk_idx, self.expert_offsets, self.perm_token, self.inv_slot, self.ws,
                    stream)
        moe_expert_ffn(s, x, self.perm_token, self.expert_offsets, w["w13"], w.get("s13"),
                       w["w2"], w.get("s2"), self.y_perm, self.ws, stream)
        moe_combine(s, self.y_perm, self.inv_slot, self.topk_w, self.y, self.ws, stream)
        return self.y

    def forward_steps(self, x, stream=None):
        """The layer as the four separate calls."""
        w, s = self.w, self.shape
        moe_route(s, x, w["wg"], w.get("bias"), self.topk_idx, self.topk_w, self.ws, stream)
        moe_permute(s, self.topk_idx, self.expert_offsets, self.perm_token, self.inv_slot, self.ws,
                    stream)
        moe_expert_ffn(s, x, self.perm_token, self.expert_offsets, w["w13"], w.get("s13"),
                       w["w2"], w.get("s2"), self.y_perm, self.ws, stream)
        moe_combine(s, self.y_perm, self.inv_slot, self.topk_w, self.y, self.ws, stream)
        return self.y
