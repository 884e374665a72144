"""focus_route_static: the routing entry point for callers that cannot allocate
device memory when they call in (an engine plugin whose memory is all pooled at
start-up, for instance).  Its Sinkhorn scratch is a fixed array inside the
library instead of a caller workspace.

Called through the C ABI with caller-owned outputs, twice in a row on different
inputs (so the second call runs on the scratch the first one left behind), and
compared with focus_route, which uses a caller workspace: same kernels and
reduction order on both sides, so membership and margins must match exactly,
the bit-exact bar the other routing tests use.  Membership is also compared with
the fp64 oracle under the near-tie rule of the other routing tests.  This file
sorts last so a run that stops at the first failure has already run every other
test; it passes alone in a fresh process too (the first call does the set-up)."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from parity import compare_membership

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
        m_np = m_static.cpu().numpy()
        np.testing.assert_array_equal(m_np, m_ws.cpu().numpy())
        np.testing.assert_array_equal(g_static.cpu().numpy(), g_ws.cpu().numpy())
        n_diff, n_near = compare_membership(wl, m_np.view(np.uint32), r, C)
        print(f"{name} seed {seed}: {n_diff} differences from the fp64 oracle "
              f"({n_near} near-ties)")


def test_static_route_without_sinkhorn_has_no_size_limit():
    """Plain top-k needs no scratch: a problem whose Sinkhorn partials would not fit
    the array runs when sinkhorn_iters = 0 and matches focus_route."""
    wl = synth.WORKLOADS["tiny"].replace(N=1 << 20, R=8, H=8, H_kv=8, K=32, top_k=2)
    p = focus.Params.from_workload(wl)
    need = 256 * -(-p.B * p.R * p.K * 4 // 256) + p.B * p.R * -(-p.N // 256) * p.K * 8
    assert need > focus.route_static_limit()
    r, C = synth.make_routing(wl, seed=2, device="cuda")
    m_static, g_static = _static_route(p, r, C)
    m_ws, g_ws = focus.route(p, r, C, margin=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(m_static.cpu().numpy(), m_ws.cpu().numpy())
    np.testing.assert_array_equal(g_static.cpu().numpy(), g_ws.cpu().numpy())
