"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every
function the header declares, sizes its workspace, and rejects bad arguments before
launching anything. Also the host-side pair accounting against the oracle."""
import ctypes
import math

import numpy as np
import pytest
import torch

import learned_centroid_gated_gb300 as focus
import oracle
from learned_centroid_gated_gb300 import pairs


# Tests that hand made-up device addresses to entry points that must reject the
# call on the host run only where no GPU is present: a regression in a check would
# then fail the test instead of launching a kernel on a bad address.
host_only = pytest.mark.skipif(torch.cuda.is_available(),
                               reason="passes made-up device addresses; host-only check")


def _params(**kw):
    base = dict(B=1, N=512, H=2, H_kv=2, d_head=64, R=1, K=4, top_k=2, w=64)
    base.update(kw)
    return focus.Params(**base)


def test_every_declared_symbol_is_exported():
    names = focus.declared_symbols()
    assert set(names) >= {"focus_route", "focus_attn_fwd", "focus_bucket", "focus_workspace_size",
                          "focus_get_status", "focus_strerror", "focus_version"}
    lib = ctypes.CDLL(focus.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_strerror():
    assert focus.version() >> 16 == 1
    assert focus.strerror(0) == "ok"
    for code in range(-8, 0):
        assert focus.strerror(code) not in ("", "unknown status")
    assert focus.strerror(-99) == "unknown status"


def test_workspace_size_valid_and_invalid():
    p = _params()
    n = focus.workspace_size(p)
    # at least the permuted copies and the fp32 long-range partial output
    assert n >= 2 * 3 * p.N * p.H * p.d_head + 4 * p.N * p.H * p.d_head
    assert focus.workspace_size(_params(N=1024)) > n
    for bad in (dict(N=0), dict(H=3, H_kv=2), dict(H_kv=2, R=3), dict(top_k=5),
                dict(K=33, top_k=1), dict(w=0), dict(d_head=96),
                dict(K=16, top_k=8, schedule=focus.SCHEDULE_SEGMENTS), dict(schedule=3),
                dict(schedule=-1), dict(sinkhorn_iters=1, sinkhorn_eps=0.0)):
        assert focus.workspace_size(_params(**bad)) == 0, bad


def _call_attn(p, q=1 << 12, k=1 << 12, v=1 << 12, r=1 << 12, C=1 << 12, mask=None, o=1 << 12,
               lse=None, ws=1 << 12, ws_bytes=None):
    P = ctypes.c_void_p
    nb = focus.workspace_size(p) if ws_bytes is None else ws_bytes
    return focus._lib.focus_attn_fwd(ctypes.byref(p.c()), P(q), P(k), P(v), P(r), P(C), P(mask),
                                     P(o), P(lse), P(ws), nb, None)


@host_only
def test_argument_errors_are_caught_on_the_host():
    p = _params()
    E = {v: k for k, v in focus.ERRORS.items()}
    assert _call_attn(p, q=None) == E["FOCUS_ERR_INVALID_ARG"]
    assert _call_attn(p, r=None) == E["FOCUS_ERR_INVALID_ARG"]   # no mask, no routing
    assert _call_attn(p, q=(1 << 12) + 2) == E["FOCUS_ERR_ALIGNMENT"]
    assert _call_attn(p, ws=(1 << 12) + 64) == E["FOCUS_ERR_ALIGNMENT"]
    assert _call_attn(p, ws_bytes=focus.workspace_size(p) - 1) == E["FOCUS_ERR_WORKSPACE"]
    assert _call_attn(_params(d_head=96)) == E["FOCUS_ERR_UNSUPPORTED"]
    assert _call_attn(_params(K=16, top_k=8, schedule=focus.SCHEDULE_SEGMENTS)) == E["FOCUS_ERR_UNSUPPORTED"]
    assert _call_attn(_params(H=4, H_kv=3)) == E["FOCUS_ERR_INVALID_ARG"]
    assert focus._lib.focus_route(None, None, None, None, None, None, 0, None) == E["FOCUS_ERR_INVALID_ARG"]


@pytest.mark.parametrize("N,w,K,top_k,R", [(1, 1, 1, 1, 1), (97, 5, 4, 2, 2), (300, 16, 6, 2, 1),
                                           (257, 300, 4, 1, 1), (200, 1, 5, 3, 1)])
def test_pair_count_matches_oracle_brute_force(N, w, K, top_k, R):
    g = torch.Generator().manual_seed(N + K)
    r = torch.randn(2, N, R, 16, generator=g)
    C = torch.randn(K, 16, generator=g)
    mask, _, _, _ = oracle.route(r, C, K=K, top_k=top_k)
    np.testing.assert_array_equal(pairs.allowed_pairs(mask, w), oracle.allowed_pairs(mask, w))


def test_window_pairs_closed_form():
    for N, w in [(1, 1), (5, 10), (10, 10), (100, 7)]:
        assert pairs.window_pairs(N, w) == sum(min(i + 1, w) for i in range(N))


def test_nseg_is_binomial():
    assert _params(K=8, top_k=2, schedule=focus.SCHEDULE_SEGMENTS).nseg == 28 == math.comb(8, 2)


def test_schedule_resolution_and_bucket_shape():
    S, G = focus.SCHEDULE_SEGMENTS, focus.SCHEDULE_GROUPS
    N = 32768
    # AUTO: smaller estimated work; on 32K tokens this is the side that measured faster
    for K, top_k, sch, nseg in [(4, 2, S, 6), (8, 2, G, 8), (8, 4, S, 70), (16, 2, G, 16),
                                (32, 2, G, 32), (16, 4, G, 16), (32, 4, G, 32), (32, 1, S, 32)]:
        rows = N * top_k if sch == G else N
        assert _params(N=N, K=K, top_k=top_k).bucket_shape() == (sch, nseg, rows), (K, top_k)
    # fewer tokens per set tip the balance towards lists; more tokens towards segments
    assert _params(N=512, K=4, top_k=2).bucket_shape()[0] == G
    assert _params(N=1 << 20, K=16, top_k=2).bucket_shape()[0] == S
    N = 512
    # explicit choices
    assert _params(K=4, top_k=2, schedule=G).bucket_shape() == (G, 4, 2 * N)
    assert _params(K=16, top_k=2, schedule=S).bucket_shape() == (S, 120, N)
    # group lists: workspace holds top_k-fold permuted copies and top_k list parts
    seg = focus.workspace_size(_params(K=4, top_k=2, schedule=S))
    grp = focus.workspace_size(_params(K=4, top_k=2, schedule=G))
    extra = 3 * 2 * N * 2 * 64 + 2 * 4 * N * 2 * 64       # one more Q/K/V copy + 2 fp32 slots
    assert grp >= seg + extra
    # 32-bit row limit counts the top_k-fold rows
    big = dict(B=1, N=1 << 24, H=64, H_kv=64, K=32, top_k=4)
    assert focus.workspace_size(_params(**big, schedule=S)) == 0       # too many sets
    assert focus.workspace_size(_params(**big)) == 0                   # 2^24 * 64 * 4 rows


@host_only
def test_host_entry_sizes_and_argument_errors():
    p = _params(H=8, H_kv=4, R=2)
    assert focus.host_workspace_size(p) > focus.workspace_size(focus.Params(**{**p.__dict__, "H": 4, "H_kv": 2, "R": 1}))
    assert focus.host_workspace_size(p, 3) == 0          # 3 does not divide H_kv
    assert focus.host_workspace_size(p, 4) == 0          # 4 does not divide R = 2
    assert focus.host_workspace_size(p, 2) > 0
    E = {v: k for k, v in focus.ERRORS.items()}
    P = ctypes.c_void_p
    h = P(1 << 12)
    n = focus.host_workspace_size(p)
    same = P(1 << 20)
    rc = focus._lib.focus_attn_fwd_host(ctypes.byref(p.c()), h, h, h, h, h, h, None, 0, P(1 << 12), n, same, same)
    assert rc == E["FOCUS_ERR_INVALID_ARG"]               # one stream for both roles
    rc = focus._lib.focus_attn_fwd_host(ctypes.byref(p.c()), h, h, h, None, h, h, None, 0, P(1 << 12), n, None, same)
    assert rc == E["FOCUS_ERR_INVALID_ARG"]               # routing inputs are required
    rc = focus._lib.focus_attn_fwd_host(ctypes.byref(p.c()), h, h, h, h, h, h, None, 0, P(1 << 12), n - 1, None, same)
    assert rc == E["FOCUS_ERR_WORKSPACE"]


@host_only
def test_backward_sizes_and_argument_errors():
    p = _params()
    n = focus.bwd_workspace_size(p)
    # permuted Q, K, V, dO (bf16) + fp32 window partials of dq, dk, dv + D
    assert n >= (4 * 2 + 3 * 4) * p.N * p.H * p.d_head + 4 * p.N * p.H
    assert focus.bwd_workspace_size(_params(K=32, top_k=4)) > n       # group lists: top_k-fold rows
    assert focus.bwd_workspace_size(_params(K=32, top_k=4, schedule=focus.SCHEDULE_SEGMENTS)) == 0
    assert focus.bwd_workspace_size(_params(d_head=96)) == 0
    E = {v: k for k, v in focus.ERRORS.items()}
    P = ctypes.c_void_p
    h = P(1 << 12)
    args = [h] * 10
    bad = list(args)
    bad[3] = None                                                      # no mask
    assert focus._lib.focus_attn_bwd(ctypes.byref(p.c()), *bad, h, n, None) == E["FOCUS_ERR_INVALID_ARG"]
    bad = list(args)
    bad[5] = None                                                      # no lse
    assert focus._lib.focus_attn_bwd(ctypes.byref(p.c()), *bad, h, n, None) == E["FOCUS_ERR_INVALID_ARG"]
    bad = list(args)
    bad[0] = P((1 << 12) + 8)                                          # misaligned q
    assert focus._lib.focus_attn_bwd(ctypes.byref(p.c()), *bad, h, n, None) == E["FOCUS_ERR_ALIGNMENT"]
    assert focus._lib.focus_attn_bwd(ctypes.byref(p.c()), *args, h, n - 1, None) == E["FOCUS_ERR_WORKSPACE"]


def test_static_route_checks_come_before_any_launch():
    """focus_route_static (no workspace): the same parameter codes as focus_route,
    and the Sinkhorn size limit before the pointer checks, so every call below is
    rejected on the host with NULL pointers and nothing can be launched."""
    E = {v: k for k, v in focus.ERRORS.items()}
    limit = focus.route_static_limit()
    assert limit == 4 << 20

    def static(p):
        return focus._lib.focus_route_static(ctypes.byref(p.c()), None, None, None, None, None)

    def ws_route(p):
        return focus._lib.focus_route(ctypes.byref(p.c()), None, None, None, None, None, 0, None)

    # Sinkhorn partials of this problem exceed the array: rejected by size first
    big = _params(N=1 << 20, H=8, H_kv=8, R=8, K=32, top_k=1, sinkhorn_iters=1)
    need = 256 * -(-8 * 32 * 4 // 256) + 8 * (big.N // 256) * 32 * 8
    assert need > limit
    assert static(big) == E["FOCUS_ERR_WORKSPACE"]
    # the same shape without Sinkhorn needs no scratch: it gets to the pointer check
    assert static(_params(N=1 << 20, H=8, H_kv=8, R=8, K=32, top_k=1)) == E["FOCUS_ERR_INVALID_ARG"]
    # parameter errors: identical codes from both routing entry points
    for bad in (dict(schedule=3), dict(N=0), dict(top_k=5), dict(d_head=96),
                dict(K=16, top_k=8, schedule=focus.SCHEDULE_SEGMENTS),
                dict(sinkhorn_iters=1, sinkhorn_eps=0.0)):
        p = _params(**bad)
        assert static(p) == ws_route(p) != 0, bad
    assert focus._lib.focus_route_static(None, None, None, None, None, None) == E["FOCUS_ERR_INVALID_ARG"]


@pytest.mark.parametrize("H_kv,R,n_groups", [(32, 1, 0), (8, 1, 0), (8, 8, 0), (16, 8, 0), (12, 1, 0),
                                              (2, 2, 0), (1, 1, 0), (16, 4, 0), (32, 1, 4), (8, 8, 2)])
def test_host_groups_cover_every_kv_head_once(H_kv, R, n_groups):
    """Groups of the host-buffer entry: consecutive, covering every KV head once,
    whole routing heads each; automatic grouping puts the smallest groups first and
    last (their copies cannot overlap compute)."""
    p = _params(H=2 * H_kv, H_kv=H_kv, R=R)
    sizes = focus.host_groups(p, n_groups)
    assert sum(sizes) == H_kv and all(s > 0 for s in sizes)
    unit = 1 if R == 1 else H_kv // R
    assert all(s % unit == 0 for s in sizes)
    if n_groups:
        assert sizes == [H_kv // n_groups] * n_groups
    elif len(sizes) >= 3:
        assert sizes[0] == sizes[-1] == min(sizes)
        if H_kv // unit >= 8:  # enough units for the edges to be smaller than the rest
            assert max(sizes) > sizes[0]
    # the workspace is sized for the largest group
    assert focus.host_workspace_size(p, n_groups) > 0


def test_window_tile_count_follows_the_skew():
    """The window pass's executed 256 x 128 tiles: ceil(span / 128) per 256-row block,
    one fewer for full blocks past the first w - 1 tokens (the two 128-row halves
    each skip one end of the band), restated per block."""
    from learned_centroid_gated_gb300 import pairs
    for N, w in ((4096, 512), (1000, 100), (300, 37), (256, 1), (777, 1024)):
        mask = np.ones((1, 1, N), np.uint32)
        _, wt = pairs.executed_tiles(mask, w)
        want = 0
        for s0 in range(0, N, 256):
            e0 = min(s0 + 256, N)
            n = -(-(e0 - max(0, s0 - w + 1)) // 128)
            want += n - (1 if (s0 >= w - 1 and e0 - s0 == 256 and n >= 2) else 0)
        assert wt == want, (N, w, wt, want)
