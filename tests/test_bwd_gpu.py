"""Backward pass (dq, dk, dv with the masks held fixed) through the C ABI vs the CPU
oracle (GPU).

Tolerance, derived from the arithmetic.  bf16 keeps an 8-bit significand, so each
rounding to bf16 has relative error <= u = 2^-8.  The kernels round P and dS to bf16
for the tensor cores and the gradients on output, and sum in fp32.  To first order an
element's error is then at most u times m, the sum of the absolute values of its
terms, which the oracle reports (mq = scale sum_j |dS_ij| |k_j|,
mk = scale sum_i |dS_ij| |q_i|, mv = sum_i P_ij |dO_i|), plus u |ref| for the output:
    |g - ref| <= 2 u m + u |ref| + 1e-6
(dq and dk are differences of large terms when P sits on few keys, so a bound relative
to |ref| alone would not hold).  The tensor core's fp32 sums (the logits and dP over
d products) are not correctly rounded: measured, they are off by up to ~2^-10 of the
sum of their terms' absolute values, which enters dS = P (dP - D) when dP ~ D; the
oracle widens m by that (d_rel = 1/4, i.e. 2^-10 in units of u).  Two kinds of check:
  kernel parity   the GPU backward receives the oracle's forward output (rounded to
                  bf16, as the API takes it) and LSE, and the oracle forms D = dO . o
                  from that same bf16 o; every gradient row of small problems.
  end to end      GPU forward, then GPU backward, against the oracle's exact
                  D = sum_j P_ij dP_ij.  The forward output's own error (its P in bf16
                  and its output rounding: 2 u of the magnitude of its terms) enters
                  D = dO . o and through dS = P (dP - D) every gradient; the oracle
                  widens m by that (d_rel = 2).
The 32K-token layer checks sampled rows and keys of one head end to end, and the sum
rules on every head."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import mask_np

focus = pytest.importorskip("learned_centroid_gated_gb300")

pytestmark = pytest.mark.gpu

U = 2.0 ** -8       # bf16 unit roundoff
UNITS = 2           # first-order bound, doubled
SUM_REL_UNITS = 0.25  # tensor-core fp32 sums: 2^-10 of their terms' magnitude, in units of u
O_REL_UNITS = 2.0     # end to end: the forward output's error, in units of u of its terms


def _check(name, g, ref, mag):
    g = g.double().cpu().numpy() if hasattr(g, "cpu") else g
    err = np.abs(g - ref)
    bound = UNITS * U * mag + U * np.abs(ref) + 1e-6
    worst = float((err / bound).max())
    assert np.isfinite(g).all(), name
    assert worst <= 1.0, f"{name}: max err/bound = {worst:.3f} (max err {err.max():.3e})"
    return worst


def _inputs(wl, seed, schedule=0):
    x = synth.make_inputs(wl, seed=seed, device="cuda")
    p = focus.Params.from_workload(wl, schedule=schedule)
    mask, _ = focus.route(p, x["r"], x["C"])
    g = torch.Generator(device="cpu").manual_seed(seed + 100)
    d_o = torch.randn(x["q"].shape, generator=g).to(torch.bfloat16).cuda()
    return x, p, mask, d_o


def _run(wl, seed=0, schedule=0):
    """GPU forward, then GPU backward."""
    x, p, mask, d_o = _inputs(wl, seed, schedule)
    o, lse = focus.attn_fwd(p, x["q"], x["k"], x["v"], mask=mask)
    dq, dk, dv = focus.attn_bwd(p, x["q"], x["k"], x["v"], mask, o, lse, d_o)
    torch.cuda.synchronize()
    return x, p, mask, o, lse, d_o, (dq, dk, dv)


SMALL = {
    "tiny": synth.WORKLOADS["tiny"],
    "ragged_gqa3": synth.WORKLOADS["tiny"].replace(N=300, H=3, H_kv=1, K=5, top_k=2, w=37),
    "routing_per_kv_group_d128_b2": synth.WORKLOADS["tiny"].replace(
        B=2, N=1000, H=4, H_kv=2, R=2, d_head=128, K=6, top_k=3, w=100),
    "window_covers_all": synth.WORKLOADS["tiny"].replace(N=700, w=900, d_head=128),
    "one_group": synth.WORKLOADS["tiny"].replace(N=513, K=1, top_k=1, d_head=128),
    "topk_equals_K": synth.WORKLOADS["tiny"].replace(N=640, K=4, top_k=4),
    "unit_window_top1": synth.WORKLOADS["tiny"].replace(N=1200, K=8, top_k=1, w=1),
    "single_token": synth.WORKLOADS["tiny"].replace(N=1),
    "many_segments_K32": synth.WORKLOADS["tiny"].replace(N=3000, K=32, top_k=2, w=50),
    "gqa4_R8_small": synth.WORKLOADS["gqa_128k"].replace(N=2048, w=128),
    "gpt2_layer": synth.WORKLOADS["gpt2_layer"],
    "K16_top3_gqa": synth.WORKLOADS["tiny"].replace(N=1500, H=8, H_kv=2, R=2, d_head=128, K=16,
                                                    top_k=3, w=100),
}


SCHEDULES = {"segments": focus.SCHEDULE_SEGMENTS, "groups": focus.SCHEDULE_GROUPS}


@pytest.mark.parametrize("schedule", list(SCHEDULES))
@pytest.mark.parametrize("name", list(SMALL))
def test_backward_kernel_parity_all_rows(name, schedule):
    wl = SMALL[name]
    x, p, mask, d_o = _inputs(wl, seed=7, schedule=SCHEDULES[schedule])
    m = mask_np(mask)
    B, N, H, d = x["q"].shape
    o_ref, lse_ref = oracle.attn(x["q"], x["k"], x["v"], m, w=wl.w, scale=p.scale)
    o16 = torch.from_numpy(o_ref).reshape(B, N, H, d).to(torch.bfloat16)
    lse32 = torch.from_numpy(lse_ref).reshape(B, N, H).permute(0, 2, 1).contiguous().float()
    dq, dk, dv = focus.attn_bwd(p, x["q"], x["k"], x["v"], mask, o16.cuda(), lse32.cuda(), d_o)
    rq, rk, rv, mq, mk, mv = oracle.attn_bwd(x["q"], x["k"], x["v"], m, d_o, w=wl.w, scale=p.scale,
                                             o_for_D=o16, magnitudes=True, d_rel=SUM_REL_UNITS)
    wq = _check("dq", dq.reshape(B * N, H, d), rq, mq)
    wk = _check("dk", dk.reshape(B * N, wl.H_kv, d), rk, mk)
    wv = _check("dv", dv.reshape(B * N, wl.H_kv, d), rv, mv)
    print(f"{name} ({schedule}): err/bound dq {wq:.2f} dk {wk:.2f} dv {wv:.2f}")


@pytest.mark.parametrize("name", ["tiny", "routing_per_kv_group_d128_b2", "many_segments_K32",
                                  "gqa4_R8_small"])
def test_backward_after_gpu_forward_all_rows(name):
    wl = SMALL[name]
    x, p, mask, o, lse, d_o, (dq, dk, dv) = _run(wl, seed=8)
    rq, rk, rv, mq, mk, mv = oracle.attn_bwd(x["q"], x["k"], x["v"], mask_np(mask), d_o, w=wl.w,
                                             scale=p.scale, magnitudes=True, d_rel=O_REL_UNITS)
    B, N, H, d = x["q"].shape
    wq = _check("dq", dq.reshape(B * N, H, d), rq, mq)
    wk = _check("dk", dk.reshape(B * N, wl.H_kv, d), rk, mk)
    wv = _check("dv", dv.reshape(B * N, wl.H_kv, d), rv, mv)
    print(f"{name} end to end: err/bound dq {wq:.2f} dk {wk:.2f} dv {wv:.2f}")


def test_backward_is_deterministic():
    wl = SMALL["routing_per_kv_group_d128_b2"]
    x, p, mask, o, lse, d_o, (dq, dk, dv) = _run(wl, seed=3)
    dq, dk, dv = dq.clone(), dk.clone(), dv.clone()
    dq2, dk2, dv2 = focus.attn_bwd(p, x["q"], x["k"], x["v"], mask, o, lse, d_o)
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)


def test_backward_full_size_sampled_rows_and_sum_rules():
    """32K tokens, 32 heads, d = 128 (the benchmark's layer), end to end: dq of 256
    sampled query rows and dk, dv of 256 sampled keys of head 0 against the oracle; on every head,
    sum_j dk_j ~ 0 and sum_j dv_j ~ sum_i dO_i (up to the bf16 rounding of the
    gradients)."""
    wl = synth.WORKLOADS["mha7b_32k"]
    x, p, mask, o, lse, d_o, (dq, dk, dv) = _run(wl, seed=0)
    rows = synth.sample_queries(wl.N, 256, wl.w, seed=5)
    keys = synth.sample_queries(wl.N, 256, wl.w, seed=6)
    rq, rk, rv, mq, mk, mv = oracle.attn_bwd(x["q"], x["k"], x["v"], mask_np(mask), d_o, w=wl.w,
                                             scale=p.scale, rows=rows, keys=keys, heads=[0],
                                             magnitudes=True, d_rel=O_REL_UNITS)
    ridx = torch.as_tensor(np.asarray(rows), device="cuda")
    kidx = torch.as_tensor(np.asarray(keys), device="cuda")
    wq = _check("dq", dq[0, ridx][:, [0]], rq, mq)
    wk = _check("dk", dk[0, kidx][:, [0]], rk[:, [0]], mk[:, [0]])
    wv = _check("dv", dv[0, kidx][:, [0]], rv[:, [0]], mv[:, [0]])
    print(f"32K end to end: err/bound dq {wq:.2f} dk {wk:.2f} dv {wv:.2f}")
    sdk = dk.double().sum(dim=1)                       # [B, H_kv, d]
    sdv = dv.double().sum(dim=1)
    sdo = d_o.double().sum(dim=1)
    adk = dk.double().abs().sum(dim=1)
    assert (sdk.abs() <= 1e-2 * adk + 1e-3).all()
    assert ((sdv - sdo).abs() <= 2e-2 * sdo.abs() + 2.0).all()


def test_backward_group_lists_35960_sets_end_to_end():
    """K = 32, top_k = 4 (35960 exact sets: group lists only), 8K tokens, GQA 8/2,
    d = 128: GPU forward then GPU backward, every row."""
    wl = synth.WORKLOADS["tiny"].replace(N=8192, H=8, H_kv=2, R=1, d_head=128, K=32, top_k=4, w=256)
    x, p, mask, o, lse, d_o, (dq, dk, dv) = _run(wl, seed=9)
    assert p.bucket_shape()[0] == focus.SCHEDULE_GROUPS
    rq, rk, rv, mq, mk, mv = oracle.attn_bwd(x["q"], x["k"], x["v"], mask_np(mask), d_o, w=wl.w,
                                             scale=p.scale, magnitudes=True, d_rel=O_REL_UNITS)
    B, N, H, d = x["q"].shape
    wq = _check("dq", dq.reshape(B * N, H, d), rq, mq)
    wk = _check("dk", dk.reshape(B * N, wl.H_kv, d), rk, mk)
    wv = _check("dv", dv.reshape(B * N, wl.H_kv, d), rv, mv)
    print(f"K32 top4 8K end to end: err/bound dq {wq:.2f} dk {wk:.2f} dv {wv:.2f}")
