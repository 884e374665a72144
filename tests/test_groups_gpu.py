"""Group-list schedule (one position-ordered list per group, a key counted only in
the list of the lowest group it shares with the query) vs the CPU oracle (GPU).

The oracle knows nothing of schedules: it evaluates the union set A_i directly, so
the same oracle output must come out of either schedule.  Includes settings the
exact-set segments cannot run at all (C(32, 4) = 35960 sets)."""
import itertools

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import compare_outputs, mask_np

focus = pytest.importorskip("learned_centroid_gated_gb300")

pytestmark = pytest.mark.gpu

G = focus.SCHEDULE_GROUPS
TINY = synth.WORKLOADS["tiny"]

CASES = {
    # name: (workload, schedule); AUTO only where C(K, top_k) > 1024 forces group lists
    "tiny_groups": (TINY, G),
    "K16_top2": (TINY.replace(N=3000, K=16, top_k=2, w=50), G),
    "K32_top4_auto": (TINY.replace(N=2500, K=32, top_k=4, w=64, d_head=128), 0),
    "K16_top3_gqa_b2": (TINY.replace(B=2, N=1500, H=8, H_kv=2, R=2, d_head=128, K=16, top_k=3,
                                     w=100), G),
    "topk_equals_K": (TINY.replace(N=700, K=8, top_k=8), G),
    "top1_groups": (TINY.replace(N=1100, K=6, top_k=1, w=16), G),
    "single_token": (TINY.replace(N=1, K=16, top_k=2), G),
    "window_covers_all": (TINY.replace(N=600, w=700, K=16, top_k=2), G),
    "sinkhorn_K16": (TINY.replace(N=2000, K=16, top_k=2, sinkhorn_iters=4, sinkhorn_eps=0.5,
                                  w=128), G),
    "K32_top2_ragged": (TINY.replace(N=3001, H=3, H_kv=1, K=32, top_k=2, w=37), G),
}


def _run(wl, schedule, seed=0, rows=None, heads=None):
    x = synth.make_inputs(wl, seed=seed, device="cuda")
    p = focus.Params.from_workload(wl, schedule=schedule)
    assert p.bucket_shape()[0] == G
    mask, _ = focus.route(p, x["r"], x["C"])
    o, lse = focus.attn_fwd(p, x["q"], x["k"], x["v"], x["r"], x["C"])
    ws = focus._default_ws[str(x["q"].device)].buf
    assert focus.get_status(ws) == 0
    m = mask_np(mask)
    o_ref, lse_ref = oracle.attn(x["q"], x["k"], x["v"], m, w=wl.w, scale=p.scale,
                                 rows=rows, heads=heads)
    return compare_outputs(o, lse, o_ref, lse_ref, rows, heads)


@pytest.mark.parametrize("name", list(CASES))
def test_group_schedule_all_rows(name):
    wl, schedule = CASES[name]
    errs = _run(wl, schedule, seed=11)
    print(f"{name}: max|dO|={errs[0]:.2e} max rel dLSE={errs[1]:.2e}")


@pytest.mark.parametrize("name", ["tiny_groups", "K32_top4_auto", "K16_top3_gqa_b2"])
def test_group_lists_are_stable_per_group(name):
    """List g = the ascending positions of the tokens whose mask has bit g."""
    wl, schedule = CASES[name]
    r, C = synth.make_routing(wl, seed=1, device="cuda")
    p = focus.Params.from_workload(wl, schedule=schedule)
    mask, _ = focus.route(p, r, C)
    perm, seg = focus.bucket(p, mask)
    assert perm.shape[-1] == wl.N * wl.top_k and seg.shape[-1] == wl.K + 1
    m = mask_np(mask).astype(np.int64)
    perm, seg = perm.cpu().numpy(), seg.cpu().numpy()
    for b, rho in itertools.product(range(wl.B), range(wl.R)):
        lists = [np.nonzero((m[b, rho] >> g) & 1)[0] for g in range(wl.K)]
        counts = np.array([len(x) for x in lists])
        np.testing.assert_array_equal(seg[b, rho], np.concatenate([[0], np.cumsum(counts)]))
        np.testing.assert_array_equal(perm[b, rho], np.concatenate(lists))


def test_both_schedules_agree_with_each_other():
    """Same inputs, both schedules: each matches the oracle, and the two agree to
    within the sum of their tolerances."""
    wl = TINY.replace(N=2048, H=4, H_kv=4, K=8, top_k=3, w=96, d_head=128)  # C(8,3) = 56
    x = synth.make_inputs(wl, seed=21, device="cuda")
    outs = []
    for sch in (focus.SCHEDULE_SEGMENTS, G):
        p = focus.Params.from_workload(wl, schedule=sch)
        o, lse = focus.attn_fwd(p, x["q"], x["k"], x["v"], x["r"], x["C"])
        outs.append((o.float().clone(), lse.clone()))
    assert (outs[0][0] - outs[1][0]).abs().max().item() < 2e-2
    assert ((outs[0][1] - outs[1][1]).abs() / outs[0][1].abs().clamp_min(1)).max().item() < 2e-3


def test_group_schedule_bad_mask_raises_bounds_without_fault():
    wl = TINY.replace(K=16, top_k=2)
    p = focus.Params.from_workload(wl, schedule=G)
    x = synth.make_inputs(wl, seed=2, device="cuda")
    bad = torch.full((1, 1, wl.N), 0b0111, dtype=torch.int32, device="cuda")
    ws = focus.Workspace("cuda").get(p)
    focus.attn_fwd(p, x["q"], x["k"], x["v"], mask=bad, ws=ws)
    assert focus.get_status(ws) == -6
    o, _ = focus.attn_fwd(p, x["q"], x["k"], x["v"], x["r"], x["C"], ws=ws)
    assert focus.get_status(ws) == 0 and torch.isfinite(o.float()).all()


def test_group_schedule_full_size_sampled_rows():
    """32K tokens, 32 heads, d = 128, K = 32, top_k = 4: the exact-set schedule
    would need 35960 segments; the group lists hold 4 x 32768 rows per head."""
    wl = synth.WORKLOADS["mha7b_32k"].replace(K=32, top_k=4)
    rows = synth.sample_queries(wl.N, 256, wl.w, seed=5)
    errs = _run(wl, 0, seed=0, rows=rows, heads=[0, 17])
    print(f"K32 top4 32K: max|dO|={errs[0]:.2e} max rel dLSE={errs[1]:.2e}")
