"""moe_route_noalloc: the router for callers that cannot allocate device memory (for instance a
plugin whose host process owns every device allocation and lends it no scratch, or a service
that fixes its device memory budget at start-up). It keeps its logits in a fixed device array
inside the library instead of a caller-provided workspace.

Checked through the C ABI against moe_route (which uses a workspace) on the same inputs, with
two calls in a row so that the second call runs over the first call's leftover scratch. This
file is collected last on purpose, and it works alone in a fresh process as well."""
import numpy as np
import pytest

import routed_expert_ffn_moe_gb300 as moe
import synth
from gpu_helpers import TOL_TOPK_W, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from routed_expert_ffn_moe_gb300 import build
    build.build()
    moe.load()


def _router_inputs(cfg):
    t = torch()
    x = synth._dev_normal(t.empty(cfg.T, cfg.d, dtype=t.bfloat16, device="cuda"), cfg.seed,
                          synth.STREAM_X, synth.SIGMA_X)
    wg = synth._dev_normal(t.empty(cfg.E, cfg.d, dtype=t.bfloat16, device="cuda"), cfg.seed,
                           synth.STREAM_WG, synth.SIGMA_W)
    b = synth.host_bias(cfg)
    bias = t.from_numpy(b).cuda() if b is not None else None
    return x, wg, bias


def _fill_scratch_with_a_larger_call():
    """A call that covers the whole scratch array (T*E = 4096*256 = 2^20 logits), so that the
    checked calls after it run over leftover values they did not write."""
    t = torch()
    cfg = synth.get_config("skewed_prefill")
    x, wg, bias = _router_inputs(cfg)
    s = moe.shape_of(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.n_shared, cfg.wdtype)
    idx = t.empty(cfg.T, cfg.k, dtype=t.int32, device="cuda")
    w = t.empty(cfg.T, cfg.k, dtype=t.float32, device="cuda")
    moe.moe_route_noalloc(s, x, wg, bias, idx, w)


def route_both(cfg, x, wg, bias):
    t = torch()
    s = moe.shape_of(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.n_shared, cfg.wdtype)
    ws = t.empty(moe.moe_workspace_size(s), dtype=t.uint8, device="cuda")
    idx_ws = t.empty(cfg.T, cfg.k, dtype=t.int32, device="cuda")
    w_ws = t.empty(cfg.T, cfg.k, dtype=t.float32, device="cuda")
    moe.moe_route(s, x, wg, bias, idx_ws, w_ws, ws)
    _fill_scratch_with_a_larger_call()
    outs = []
    for _ in range(2):  # two calls in a row share the library's scratch array
        idx = t.full((cfg.T, cfg.k), -7, dtype=t.int32, device="cuda")
        w = t.full((cfg.T, cfg.k), -7.0, dtype=t.float32, device="cuda")
        moe.moe_route_noalloc(s, x, wg, bias, idx, w)
        outs.append((idx, w))
    t.cuda.synchronize()
    return (idx_ws.cpu().numpy(), w_ws.cpu().numpy()), [(i.cpu().numpy(), w.cpu().numpy())
                                                          for i, w in outs]


@pytest.mark.parametrize("name,over", [("tiny", {"T": 37}), ("v3_decode", {}),
                                       ("skewed_prefill", {}), ("v4pro_decode", {})])
def test_noalloc_router_matches_workspace_router(name, over):
    # the same bits as moe_route: the expert choice and the gate weights alike
    cfg = synth.get_config(name, **over)
    x, wg, bias = _router_inputs(cfg)
    (idx_ref, w_ref), calls = route_both(cfg, x, wg, bias)
    for idx, w in calls:
        np.testing.assert_array_equal(idx, idx_ref)
        np.testing.assert_array_equal(w.view(np.int32), w_ref.view(np.int32))
        assert np.abs(w - w_ref).max() <= TOL_TOPK_W


def test_noalloc_router_rejects_shapes_beyond_its_scratch():
    # T*E = 4097 * 256 > 2^20: refused on the host before any launch
    s = moe.shape_of(4097, 7168, 256, 8, 2048, 1, "bf16")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_route_noalloc(s, 0x7F0000000000, 0x7F0000000000, None, 0x7F0000000000,
                              0x7F0000000000, stream=0)
    assert ei.value.status == -1 and "built-in scratch" in str(ei.value)
