"""Routing and bucketing kernels vs the CPU oracle (GPU)."""
import itertools

import numpy as np
import pytest
import torch

import synth
from parity import NEAR_TIE, compare_membership, mask_np, route_oracle

focus = pytest.importorskip("learned_centroid_gated_gb300")

pytestmark = pytest.mark.gpu

ALL = list(synth.WORKLOADS)


@pytest.mark.parametrize("name", ALL)
def test_membership_matches_oracle(name):
    wl = synth.WORKLOADS[name]
    r, C = synth.make_routing(wl, seed=0, device="cuda")
    p = focus.Params.from_workload(wl)
    mask, margin = focus.route(p, r, C, margin=True)
    m = mask_np(mask)
    assert np.all(np.vectorize(lambda x: bin(int(x)).count("1"))(m[:, :, :4096]) == wl.top_k)
    n_diff, n_near = compare_membership(wl, m, r, C)
    print(f"{name}: {n_diff} membership differences, {n_near} near-ties (< {NEAR_TIE})")
    if wl.sinkhorn_iters == 0:
        # same decision precision: fp32 fused multiply-add scores -> bit-exact
        m32, marg32, _, _ = route_oracle(wl, r, C, score_fp32=True)
        np.testing.assert_array_equal(m, m32)
        np.testing.assert_allclose(margin.cpu().numpy(), marg32, rtol=0, atol=1e-5)


@pytest.mark.parametrize("K,top_k,T,eps,N,R", [
    (1, 1, 0, 1.0, 100, 1), (5, 5, 0, 1.0, 100, 2), (32, 2, 0, 1.0, 3000, 1),
    (6, 2, 5, 0.5, 2000, 2), (8, 1, 1, 2.0, 777, 1), (4, 2, 3, 1.0, 1, 1)])
def test_membership_edge_cases(K, top_k, T, eps, N, R):
    wl = synth.WORKLOADS["tiny"].replace(N=N, K=K, top_k=top_k, sinkhorn_iters=T, sinkhorn_eps=eps,
                                         R=R, H=2 * R, H_kv=R)
    r, C = synth.make_routing(wl, seed=3, device="cuda")
    p = focus.Params.from_workload(wl)
    mask, _ = focus.route(p, r, C)
    compare_membership(wl, mask_np(mask), r, C)


def _colex_rank_table(K, top_k):
    subsets = sorted(itertools.combinations(range(K), top_k), key=lambda s: tuple(reversed(s)))
    return {sum(1 << g for g in s): i for i, s in enumerate(subsets)}


@pytest.mark.parametrize("name", ["tiny", "gpt2_layer", "gqa_128k"])
def test_bucketing_is_stable_sort_by_mask_value(name):
    wl = synth.WORKLOADS[name]
    r, C = synth.make_routing(wl, seed=1, device="cuda")
    p = focus.Params.from_workload(wl, schedule=focus.SCHEDULE_SEGMENTS)
    mask, _ = focus.route(p, r, C)
    perm, seg = focus.bucket(p, mask)
    m = mask_np(mask)
    table = _colex_rank_table(wl.K, wl.top_k)
    perm, seg = perm.cpu().numpy(), seg.cpu().numpy()
    for b, rho in itertools.product(range(wl.B), range(wl.R)):
        rank = np.array([table[int(x)] for x in m[b, rho]])
        np.testing.assert_array_equal(perm[b, rho], np.argsort(rank, kind="stable"))
        counts = np.bincount(rank, minlength=len(table))
        np.testing.assert_array_equal(seg[b, rho], np.concatenate([[0], np.cumsum(counts)]))


def test_bad_mask_raises_bounds_status_without_fault():
    wl = synth.WORKLOADS["tiny"]
    p = focus.Params.from_workload(wl, schedule=focus.SCHEDULE_SEGMENTS)
    mask = torch.full((1, 1, wl.N), 0b0111, dtype=torch.int32, device="cuda")  # 3 bits, top_k=2
    ws = focus.Workspace("cuda").get(p)
    focus.bucket(p, mask, ws=ws)
    assert focus.get_status(ws) == -6
    good, _ = focus.route(p, *synth.make_routing(wl, device="cuda"), ws=ws)
    assert focus.get_status(ws) == 0
