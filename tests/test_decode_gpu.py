"""Decode step (newest token of each sequence over its cache) through the C ABI vs
the CPU oracle's last row, on the same union set as the forward pass."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import LSE_RTOL, O_ATOL, mask_np

focus = pytest.importorskip("learned_centroid_gated_gb300")

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": synth.WORKLOADS["tiny"],
    "gpt2_layer": synth.WORKLOADS["gpt2_layer"],
    "mha7b_32k": synth.WORKLOADS["mha7b_32k"],
    "gqa_128k": synth.WORKLOADS["gqa_128k"],
    "extreme_1m": synth.WORKLOADS["extreme_1m"],
    "mqa16_b2": synth.WORKLOADS["tiny"].replace(B=2, N=3000, H=16, H_kv=1, d_head=128, K=6, top_k=2, w=100),
    "gqa3_ragged_heads": synth.WORKLOADS["tiny"].replace(N=5000, H=6, H_kv=2, R=2, d_head=64, K=5, top_k=2, w=77),
    "single_token": synth.WORKLOADS["tiny"].replace(N=1),
    "window_covers_all": synth.WORKLOADS["tiny"].replace(N=700, w=4096),
    "one_group": synth.WORKLOADS["tiny"].replace(N=1025, K=1, top_k=1, w=16),
}


@pytest.mark.parametrize("name", list(CASES))
def test_decode_matches_oracle_last_row(name):
    wl = CASES[name]
    x = synth.make_inputs(wl, seed=7, device="cuda")
    p = focus.Params.from_workload(wl)
    mask, _ = focus.route(p, x["r"], x["C"])
    q_new = x["q"][:, wl.N - 1].contiguous()
    o, lse = focus.decode(p, q_new, x["k"], x["v"], mask)
    rows = np.array([b * wl.N + wl.N - 1 for b in range(wl.B)])
    o_ref, lse_ref = oracle.attn(x["q"], x["k"], x["v"], mask_np(mask), w=wl.w, rows=rows)
    o_g = o.float().double().cpu().numpy()
    l_g = lse.double().cpu().numpy()
    err_o = np.abs(o_g - o_ref).max()
    err_l = (np.abs(l_g - lse_ref) / np.maximum(1.0, np.abs(lse_ref))).max()
    print(f"{name}: max|dO|={err_o:.2e} max rel dLSE={err_l:.2e}")
    assert err_o <= O_ATOL and err_l <= LSE_RTOL


def test_decode_equals_forward_last_row():
    """The decode step and the forward pass agree on the last row."""
    wl = synth.WORKLOADS["tiny"].replace(N=2000, H=4, H_kv=2, d_head=128)
    x = synth.make_inputs(wl, seed=8, device="cuda")
    p = focus.Params.from_workload(wl)
    mask, _ = focus.route(p, x["r"], x["C"])
    o_f, l_f = focus.attn_fwd(p, x["q"], x["k"], x["v"], mask=mask)
    o_d, l_d = focus.decode(p, x["q"][:, -1].contiguous(), x["k"], x["v"], mask)
    assert (o_f[:, -1].float() - o_d.float()).abs().max().item() <= 1e-2
    assert (l_f[:, :, -1] - l_d).abs().max().item() <= 1e-4
