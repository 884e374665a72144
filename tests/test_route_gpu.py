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


def test_nonfinite_routing_inputs_raise_status_without_fault():
    """A NaN routing vector and an infinite component: the kernel raises
    FOCUS_ERR_NONFINITE, every token still gets exactly top_k groups (a NaN key ranks
    below every number, ties to the lower group), the finite tokens match the oracle,
    and the forward pass that routes internally completes with finite outputs."""
    wl = synth.WORKLOADS["tiny"].replace(N=700, K=6, top_k=2, R=2, H=4, H_kv=2)
    r, C = synth.make_routing(wl, seed=7, device="cuda")
    r[0, 5, 0, :] = float("nan")      # every score of token 5 (routing head 0) is NaN
    r[0, 9, 1, 3] = float("inf")      # token 9 (routing head 1): scores are +-inf
    p = focus.Params.from_workload(wl)
    ws = focus.Workspace("cuda").get(p)
    mask, _ = focus.route(p, r, C, ws=ws)
    assert focus.get_status(ws) == -8
    m = mask_np(mask)
    assert m[0, 0, 5] == (1 << wl.top_k) - 1
    c3 = C[:, 3].cpu().numpy()
    key = np.where(c3 > 0, np.inf, -np.inf)
    want = np.argsort(-key, kind="stable")[:wl.top_k]
    assert m[0, 1, 9] == sum(1 << int(g) for g in want)
    bits = np.vectorize(lambda v: bin(int(v)).count("1"))(m)
    assert (bits == wl.top_k).all()
    finite = torch.isfinite(r).all(dim=-1).cpu().numpy()  # [B, N, R]
    m64, marg64, _, _ = route_oracle(wl, torch.nan_to_num(r, nan=0.0, posinf=0.0), C)
    ok = finite.transpose(0, 2, 1) & (marg64 >= NEAR_TIE)
    np.testing.assert_array_equal(m[ok], m64[ok])
    x = synth.make_inputs(wl, seed=7, device="cuda")
    o, lse = focus.attn_fwd(p, x["q"], x["k"], x["v"], r, C, ws=ws)
    assert focus.get_status(ws) == -8
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    # the next call on clean inputs clears the status
    focus.route(p, *synth.make_routing(wl, seed=7, device="cuda"), ws=ws)
    assert focus.get_status(ws) == 0


def test_nonfinite_routing_with_sinkhorn_is_well_defined():
    """With Sinkhorn, a NaN vector spreads through the column potentials of its
    (b, routing head): every token of that routing head ranks all-NaN keys and gets
    groups 0..top_k-1; the other routing head is untouched and matches the oracle."""
    wl = synth.WORKLOADS["tiny"].replace(N=900, K=5, top_k=2, R=2, H=4, H_kv=2, sinkhorn_iters=2)
    r, C = synth.make_routing(wl, seed=8, device="cuda")
    r[0, 17, 0, 2] = float("nan")
    p = focus.Params.from_workload(wl)
    ws = focus.Workspace("cuda").get(p)
    mask, _ = focus.route(p, r, C, ws=ws)
    assert focus.get_status(ws) == -8
    m = mask_np(mask)
    assert (m[0, 0] == (1 << wl.top_k) - 1).all()
    wl1 = wl.replace(R=1, H=2, H_kv=1)
    r1 = r[:, :, 1:2].contiguous()
    compare_membership(wl1, m[:, 1:2], r1, C)
