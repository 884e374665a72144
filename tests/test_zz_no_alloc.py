"""focus_route_static: the routing entry point for callers that cannot allocate
device memory when they call in (its scratch is a fixed array inside the library).

Called through the C ABI with caller-owned outputs, twice in a row on different
inputs (so the second call runs on scratch the first one left behind), and
compared with focus_route, which uses a caller workspace. Same kernels and
reduction order on both sides, so membership and margins must match exactly,
the same bit-exact bar the other routing tests use.  This file sorts last so a
run that stops at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import synth

focus = pytest.importorskip("learned_centroid_gated_gb300")

pytestmark = pytest.mark.gpu


def _static_route(p, r, C):
    mask = torch.empty(p.B, p.R, p.N, dtype=torch.int32, device=r.device)
    margin = torch.empty(p.B, p.R, p.N, dtype=torch.float32, device=r.device)
    stream = torch.cuda.current_stream()
    rc = focus._lib.focus_route_static(ctypes.byref(p.c()), ctypes.c_void_p(r.data_ptr()),
                                       ctypes.c_void_p(C.data_ptr()),
                                       ctypes.c_void_p(mask.data_ptr()),
                                       ctypes.c_void_p(margin.data_ptr()),
                                       ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0, focus.strerror(rc)
    return mask, margin


@pytest.mark.parametrize("name", ["gpt2_layer", "tiny"])
def test_static_scratch_route_matches_workspace_route(name):
    wl = synth.WORKLOADS[name]
    if wl.sinkhorn_iters == 0:
        wl = wl.replace(sinkhorn_iters=2, R=2, H=4, H_kv=2)  # exercise the scratch
    p = focus.Params.from_workload(wl)
    for seed in (0, 1):  # two calls in a row on different inputs
        r, C = synth.make_routing(wl, seed=seed, device="cuda")
        m_static, g_static = _static_route(p, r, C)
        m_ws, g_ws = focus.route(p, r, C, margin=True)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(m_static.cpu().numpy(), m_ws.cpu().numpy())
        np.testing.assert_array_equal(g_static.cpu().numpy(), g_ws.cpu().numpy())


def test_static_scratch_rejects_problems_beyond_its_size():
    wl = synth.WORKLOADS["extreme_1m"].replace(K=32, top_k=1, R=8, sinkhorn_iters=1)
    p = focus.Params.from_workload(wl)
    rc = focus._lib.focus_route_static(ctypes.byref(p.c()), ctypes.c_void_p(1 << 12),
                                       ctypes.c_void_p(1 << 12), ctypes.c_void_p(1 << 12), None,
                                       None)
    assert focus.ERRORS[rc] == "FOCUS_ERR_WORKSPACE"
