"""Host-side checks of the C ABI: the library builds and loads, exports every entry point that
include/moe.h declares, sizes workspaces, and rejects bad arguments before any launch. No call
here reaches a kernel (every bad-argument case fails validation first), so no GPU is needed."""
import ctypes
import os
import re

import pytest

import routed_expert_ffn_moe_gb300 as moe
from routed_expert_ffn_moe_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.load()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert set(names) == set(moe.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n
    # and nothing else leaks out of the library (hidden visibility)
    out = os.popen(f"nm -D --defined-only {moe.lib_path()}").read()
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert {s for s in exported if s.startswith("moe_")} == set(names)


def test_library_targets_sm_103a_only():
    # the build passes exactly one -gencode, for sm_103a
    assert moe_build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_workspace_size_valid_and_invalid(lib):
    s = moe.shape_of(256, 7168, 256, 8, 2048, 1, "bf16")
    n = moe.moe_workspace_size(s)
    # holds at least the logits, gathered rows and h of this shape, and the tensor-core
    # router's tile plan and row norms
    assert n >= 256 * 256 * 4 + 256 * 8 * 7168 * 2 + 256 * 9 * 2048 * 2 + 16 + 256 * 4
    assert n % 256 == 0
    assert moe.moe_workspace_size(moe.shape_of(0, 256, 8, 2, 128)) > 0
    for bad in (moe.shape_of(16, 250, 8, 2, 128), moe.shape_of(16, 256, 8, 9, 128),
                moe.shape_of(16, 256, 0, 1, 128), moe.shape_of(16, 256, 8, 2, 100),
                moe.shape_of(16, 256, 8, 2, 128, n_shared=2), moe.shape_of(-1, 256, 8, 2, 128),
                moe.shape_of(16, 256, 2000, 2, 128), moe.shape_of(16, 256, 64, 33, 128),
                moe.MoeShape(16, 256, 8, 2, 128, 1, 7)):
        assert moe.moe_workspace_size(bad) == 0


FAKE = 0x7F0000000000  # never dereferenced: every call below fails host validation


def call(fn, *args):
    rc = getattr(moe.load(), fn)(*args)
    return rc, moe.moe_last_error_string()


def test_bad_arguments_rejected_before_launch(lib):
    s = moe.shape_of(16, 256, 8, 2, 128)
    sp = ctypes.byref(s)
    wsz = moe.moe_workspace_size(s)
    F = FAKE
    rc, msg = call("moe_route", sp, None, F, None, F, F, F, wsz, None)
    assert rc == -1 and "x is NULL" in msg
    rc, msg = call("moe_route", sp, F + 8, F, None, F, F, F, wsz, None)
    assert rc == -1 and "aligned" in msg
    rc, msg = call("moe_route", sp, F, F, None, F, F, F, wsz - 1, None)
    assert rc == -3 and "workspace" in msg
    rc, msg = call("moe_route", sp, F, F, None, F, F, F + 16, wsz, None)
    assert rc == -1 and "ws" in msg
    rc, msg = call("moe_permute", sp, F, None, F, F, F, wsz, None)
    assert rc == -1 and "expert_offsets" in msg
    rc, msg = call("moe_expert_ffn", sp, F, F, F, F, F, F, None, F, F, wsz, None)
    assert rc == -1 and "must be NULL" in msg
    s8 = moe.shape_of(16, 256, 8, 2, 128, 1, "fp8")
    rc, msg = call("moe_expert_ffn", ctypes.byref(s8), F, F, F, F, None, F, None, F, F,
                   moe.moe_workspace_size(s8), None)
    assert rc == -1 and "s13" in msg
    rc, msg = call("moe_combine", sp, F, F, F, None, F, wsz, None)
    assert rc == -1 and "y is NULL" in msg
    bad = moe.shape_of(16, 256, 8, 3, 100)
    rc, msg = call("moe_combine", ctypes.byref(bad), F, F, F, F, F, wsz, None)
    assert rc == -1 and "f=100" in msg
    rc, msg = call("moe_route", None, F, F, None, F, F, F, wsz, None)
    assert rc == -1 and "shape is NULL" in msg
    rc, msg = call("moe_check_device_status", F + 64, None)
    assert rc == -1
    # moe_forward: x, wg, bias, w13, s13, w2, s2, topk_idx, topk_w, offsets, perm, inv, y_perm, y
    fwd = [F, F, None, F, None, F, None, F, F, F, F, F, F, F]
    bad = list(fwd); bad[13] = None
    rc, msg = call("moe_forward", sp, *bad, F, wsz, None)
    assert rc == -1 and "y is NULL" in msg
    bad = list(fwd); bad[4] = F
    rc, msg = call("moe_forward", sp, *bad, F, wsz, None)
    assert rc == -1 and "must be NULL" in msg
    rc, msg = call("moe_forward", sp, *fwd, F, wsz - 1, None)
    assert rc == -3 and "workspace" in msg
    rc, msg = call("moe_selftest_bounded_wait", F, 0, None)
    assert rc == -1 and "limit_us" in msg
    rc, msg = call("moe_selftest_bounded_wait", F, 2_000_001, None)
    assert rc == -1 and "limit_us" in msg
    rc, msg = call("moe_selftest_bounded_wait", F + 16, 1000, None)
    assert rc == -1 and "ws" in msg


def test_mxfp4_arguments_rejected_before_launch(lib):
    s4 = moe.shape_of(16, 256, 8, 2, 128, 1, "mxfp4")
    sp = ctypes.byref(s4)
    wsz = moe.moe_workspace_size(s4)
    # the workspace holds x and h as two E4M3 terms plus a scale byte per 32 elements each
    slots = 16 * 3
    assert wsz >= slots * (2 * 256 + 2 * 8) + slots * (2 * 128 + 2 * 4)
    F = FAKE
    # shape, x, perm_token, offsets, w13, s13, w2, s2, y_perm, ws, ws_bytes, stream
    rc, msg = call("moe_expert_ffn", sp, F, F, F, F + 16, F, F, F, F, F, wsz, None)
    assert rc == -1 and "w13 not 32-byte aligned" in msg
    rc, msg = call("moe_expert_ffn", sp, F, F, F, F, None, F, F, F, F, wsz, None)
    assert rc == -1 and "s13 is NULL" in msg
    rc, msg = call("moe_expert_ffn", sp, F, F, F, F, F, F, F + 8, F, F, wsz, None)
    assert rc == -1 and "s2 not 16-byte aligned" in msg
    # moe_forward: x, wg, bias, w13, s13, w2, s2, topk_idx, topk_w, offsets, perm, inv, y_perm, y
    fwd = [F, F, None, F, F, F + 16, F, F, F, F, F, F, F, F]
    rc, msg = call("moe_forward", sp, *fwd, F, wsz, None)
    assert rc == -1 and "w2 not 32-byte aligned" in msg
    assert moe.moe_workspace_size(moe.MoeShape(16, 256, 8, 2, 128, 1, 3)) == 0


def test_hash_route_arguments_rejected_before_launch(lib):
    s = moe.shape_of(16, 256, 8, 2, 128)
    sp = ctypes.byref(s)
    wsz = moe.moe_workspace_size(s)
    F = FAKE
    # shape, x, wg, bias, token_ids, tid2eid, vocab, topk_idx, topk_w, ws, ws_bytes, stream
    rc, msg = call("moe_route_hash", sp, F, F, None, F, F, 0, F, F, F, wsz, None)
    assert rc == -1 and "vocab=0" in msg
    rc, msg = call("moe_route_hash", sp, F, F, None, None, F, 100, F, F, F, wsz, None)
    assert rc == -1 and "token_ids is NULL" in msg
    rc, msg = call("moe_route_hash", sp, F, F, None, F, F + 4, 100, F, F, F, wsz, None)
    assert rc == -1 and "tid2eid not 16-byte aligned" in msg
    rc, msg = call("moe_route_hash", sp, F, F, None, F, F, 100, F, F, F, wsz - 1, None)
    assert rc == -3


def test_binding_raises_moe_error(lib):
    s = moe.shape_of(16, 256, 8, 2, 128)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_route(s, None, FAKE, None, FAKE, FAKE, FAKE, stream=0, ws_bytes=10 ** 9)
    assert ei.value.status == -1


def test_product_path_never_imports_the_oracle():
    # The CUDA library's Python binding and sources do not reference the oracle.
    pkg = os.path.join(ROOT, "routed_expert_ffn_moe_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for fn in files:
            if fn.endswith((".py", ".cu", ".h", ".cuh")):
                text = open(os.path.join(dirpath, fn), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, fn
                assert "moe_oracle" not in text, fn
