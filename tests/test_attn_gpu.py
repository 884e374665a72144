"""Focus attention forward through the C ABI vs the CPU oracle (GPU).

Small problems compare every output row; the full-size workloads compare a seeded
sample of query rows (always including 0, w-1, w and N-1) in exactly the launch
configuration the benchmark times.  The oracle runs on the mask the GPU produced
(so a flipped near-tie cannot fail the output check); membership itself is
compared separately, bit-exact away from near-ties."""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import compare_membership, compare_outputs, mask_np

focus = pytest.importorskip("learned_centroid_gated_gb300")

pytestmark = pytest.mark.gpu


def _run(wl, seed=0, rows=None, heads=None, scale=0.0, use_mask_in=False, schedule=0):
    x = synth.make_inputs(wl, seed=seed, device="cuda")
    p = focus.Params.from_workload(wl, softmax_scale=scale, schedule=schedule)
    mask, _ = focus.route(p, x["r"], x["C"])
    if use_mask_in:
        o, lse = focus.attn_fwd(p, x["q"], x["k"], x["v"], mask=mask)
    else:
        o, lse = focus.attn_fwd(p, x["q"], x["k"], x["v"], x["r"], x["C"])
    ws = focus._default_ws[str(x["q"].device)].buf
    assert focus.get_status(ws) == 0
    m = mask_np(mask)
    o_ref, lse_ref = oracle.attn(x["q"], x["k"], x["v"], m, w=wl.w,
                                 scale=p.scale, rows=rows, heads=heads)
    errs = compare_outputs(o, lse, o_ref, lse_ref, rows, heads)
    return x, m, errs


SMALL = {
    "tiny": synth.WORKLOADS["tiny"],
    "gpt2_layer": synth.WORKLOADS["gpt2_layer"],
    "single_token": synth.WORKLOADS["tiny"].replace(N=1),
    "ragged_gqa3": synth.WORKLOADS["tiny"].replace(N=300, H=3, H_kv=1, K=5, top_k=2, w=37),
    "ragged_gqa3_d128": synth.WORKLOADS["tiny"].replace(N=300, H=3, H_kv=1, K=5, top_k=2, w=37,
                                                        d_head=128),
    "single_token_d128": synth.WORKLOADS["tiny"].replace(N=1, d_head=128),
    "routing_per_kv_group_d128_b2": synth.WORKLOADS["tiny"].replace(
        B=2, N=1000, H=4, H_kv=2, R=2, d_head=128, K=6, top_k=3, w=100),
    "window_covers_all": synth.WORKLOADS["tiny"].replace(N=700, w=900, d_head=128),
    "one_group": synth.WORKLOADS["tiny"].replace(N=513, K=1, top_k=1, d_head=128),
    "topk_equals_K": synth.WORKLOADS["tiny"].replace(N=640, K=4, top_k=4),
    "unit_window_top1": synth.WORKLOADS["tiny"].replace(N=1200, K=8, top_k=1, w=1),
    "sinkhorn5": synth.WORKLOADS["tiny"].replace(N=2000, sinkhorn_iters=5, sinkhorn_eps=0.5, w=128),
    "many_segments_K32": synth.WORKLOADS["tiny"].replace(N=3000, K=32, top_k=2, w=50),
    "gqa4_R8_small": synth.WORKLOADS["gqa_128k"].replace(N=2048, w=128),
    "extreme_small": synth.WORKLOADS["extreme_1m"].replace(N=4096, w=256),
}


SCHEDULES = {"segments": focus.SCHEDULE_SEGMENTS, "groups": focus.SCHEDULE_GROUPS}


@pytest.mark.parametrize("schedule", list(SCHEDULES))
@pytest.mark.parametrize("name", list(SMALL))
def test_attention_all_rows(name, schedule):
    wl = SMALL[name]
    _, _, errs = _run(wl, seed=1, schedule=SCHEDULES[schedule])
    print(f"{name} ({schedule}): max|dO|={errs[0]:.2e} max rel dLSE={errs[1]:.2e}")


@pytest.mark.parametrize("d_head", [64, 128])
@pytest.mark.parametrize("schedule", list(SCHEDULES))
def test_scores_growing_along_the_sequence(schedule, d_head):
    """Scores that grow by ~100 (log2 units) from the first keys to the last, so the
    kernels' running max lags far behind and has to be retaken mid-row (the path a
    tile whose exponentials sum past the cap takes), in the window and long-range
    passes; compared with the oracle on every row."""
    wl = synth.WORKLOADS["tiny"].replace(N=1500, w=100, K=4, top_k=2, d_head=d_head)
    x = synth.make_inputs(wl, seed=6, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(6)
    pos = torch.arange(wl.N, device="cuda", dtype=torch.float32).view(1, wl.N, 1, 1)
    q = (torch.rand(x["q"].shape, generator=g, device="cuda") + 0.5).to(torch.bfloat16)
    k = ((torch.rand(x["k"].shape, generator=g, device="cuda") + 0.5) * (1 + 5 * pos / wl.N)).to(torch.bfloat16)
    p = focus.Params.from_workload(wl, schedule=SCHEDULES[schedule])
    mask, _ = focus.route(p, x["r"], x["C"])
    o, lse = focus.attn_fwd(p, q, k, x["v"], mask=mask)
    ws = focus._default_ws[str(q.device)].buf
    assert focus.get_status(ws) == 0
    o_ref, lse_ref = oracle.attn(q, k, x["v"], mask_np(mask), w=wl.w, scale=p.scale)
    assert lse_ref.max() - lse_ref.min() > 40.0  # natural-log units: a wide range of maxima
    errs = compare_outputs(o, lse, o_ref, lse_ref)
    print(f"growing scores ({schedule}): max|dO|={errs[0]:.2e} max rel dLSE={errs[1]:.2e}")


ENGINE_CASES = {
    "extreme_small": SMALL["extreme_small"],
    "ragged_gqa3_d128": SMALL["ragged_gqa3_d128"],
    "routing_per_kv_group_d128_b2": SMALL["routing_per_kv_group_d128_b2"],
}


@pytest.mark.parametrize("engine", ["pair", "single"])
@pytest.mark.parametrize("name", list(ENGINE_CASES))
def test_both_long_range_engines(name, engine, monkeypatch):
    """FOCUS_LONG_ENGINE=pair runs the long-range pass (d = 128, exact-set segments)
    on CTA pairs; by default the one-CTA kernel runs it.  Both against the oracle."""
    if engine == "pair":
        monkeypatch.setenv("FOCUS_LONG_ENGINE", "pair")
    else:
        monkeypatch.delenv("FOCUS_LONG_ENGINE", raising=False)
    _, _, errs = _run(ENGINE_CASES[name], seed=4, schedule=focus.SCHEDULE_SEGMENTS)
    print(f"{name} ({engine}): max|dO|={errs[0]:.2e} max rel dLSE={errs[1]:.2e}")


@pytest.mark.parametrize("schedule", list(SCHEDULES))
def test_precomputed_mask_and_explicit_scale(schedule):
    wl = synth.WORKLOADS["tiny"].replace(N=777, w=33)
    _run(wl, seed=2, scale=0.05, use_mask_in=True, schedule=SCHEDULES[schedule])


@pytest.mark.parametrize("schedule", list(SCHEDULES))
def test_deterministic_across_calls(schedule):
    wl = synth.WORKLOADS["gpt2_layer"]
    x = synth.make_inputs(wl, seed=3, device="cuda")
    p = focus.Params.from_workload(wl, schedule=SCHEDULES[schedule])
    o1, l1 = focus.attn_fwd(p, x["q"], x["k"], x["v"], x["r"], x["C"])
    o1, l1 = o1.clone(), l1.clone()
    o2, l2 = focus.attn_fwd(p, x["q"], x["k"], x["v"], x["r"], x["C"])
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


HOST_CASES = {"routing_pairs_16kv": synth.WORKLOADS["tiny"].replace(
    N=700, H=16, H_kv=16, R=8, K=5, top_k=2, w=50)}


@pytest.mark.parametrize("name,n_groups", [("tiny", 0), ("gpt2_layer", 0), ("gpt2_layer", 4),
                                           ("gpt2_layer", 3), ("gqa4_R8_small", 0),
                                           ("gqa4_R8_small", 2), ("routing_pairs_16kv", 0)])
def test_host_buffer_entry_matches_device_entry(name, n_groups):
    """Grouped, copy-overlapped host entry = device entry, bit for bit (heads are
    independent problems and each head's arithmetic is the same), with equal groups
    and with the automatic unequal ones (small first and last group; groups of two
    KV heads sharing one routing head in the last case)."""
    wl = SMALL.get(name) or HOST_CASES.get(name) or synth.WORKLOADS[name]
    x = {k: v.pin_memory() for k, v in synth.make_inputs(wl, seed=4, device="cpu").items()}
    p = focus.Params.from_workload(wl)
    o_h, l_h = focus.attn_fwd_host(p, x["q"], x["k"], x["v"], x["r"], x["C"], n_groups=n_groups)
    d = {k: v.cuda() for k, v in x.items()}
    o_d, l_d = focus.attn_fwd(p, d["q"], d["k"], d["v"], d["r"], d["C"])
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())


# Full-size workloads in the benchmark's launch configuration, every head: the 32K
# layer on all of its rows, the 128K GQA layer on a seeded sample of 8192 query
# rows, the 1M-token layer on a seeded sample of 4096 (always including 0, w-1, w
# and N-1).  Membership is compared for all N tokens.  FOCUS_TEST_SAMPLES
# overrides the row count of the sampled ones.
FULL = {"mha7b_32k": None, "gqa_128k": 8192, "extreme_1m": 4096}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_rows_all_heads(name):
    wl = synth.WORKLOADS[name]
    n = FULL[name]
    rows = None
    if n is not None:
        n = int(os.environ.get("FOCUS_TEST_SAMPLES", n))
        rows = synth.sample_queries(wl.N, n, wl.w, seed=5)
    x, m, errs = _run(wl, seed=0, rows=rows)
    n_diff, n_near = compare_membership(wl, m, x["r"], x["C"])
    print(f"{name}: {wl.N if rows is None else len(rows)} rows x {wl.H} heads, "
          f"max|dO|={errs[0]:.2e} max rel dLSE={errs[1]:.2e}, "
          f"membership differences {n_diff} (near-ties {n_near}) over {wl.N} tokens")
