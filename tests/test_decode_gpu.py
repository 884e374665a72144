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
    "gqa8_K16_top3": synth.WORKLOADS["tiny"].replace(N=20000, H=32, H_kv=4, R=4, d_head=128, K=16, top_k=3,
                                                     w=300),
    "gqa3_d128_odd_N": synth.WORKLOADS["tiny"].replace(B=3, N=4099, H=12, H_kv=4, d_head=128, K=4, top_k=1,
                                                       w=1000),
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


def test_decode_is_deterministic_and_graph_replay_equals_eager():
    """Two eager calls agree bit for bit; the step captured in a CUDA graph (the
    combine kernel is a programmatic dependent launch of the split kernel) replays to
    the same bits on new inputs copied into the captured buffers."""
    wl = synth.WORKLOADS["tiny"].replace(N=9000, H=8, H_kv=2, d_head=128, K=8, top_k=2, w=200)
    p = focus.Params.from_workload(wl)
    x = synth.make_inputs(wl, seed=11, device="cuda")
    mask, _ = focus.route(p, x["r"], x["C"])
    q_new = x["q"][:, -1].contiguous()
    o1, l1 = focus.decode(p, q_new, x["k"], x["v"], mask)
    o2, l2 = focus.decode(p, q_new, x["k"], x["v"], mask)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ws = torch.empty(focus.decode_workspace_size(p), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(o1)
    lse = torch.empty_like(l1)
    kc, vc, mk = x["k"].clone(), x["v"].clone(), mask.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # first call (kernel attributes) outside capture
        focus.decode(p, q_new, kc, vc, mk, out=o, lse=lse, ws=ws, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        focus.decode(p, q_new, kc, vc, mk, out=o, lse=lse, ws=ws, stream=torch.cuda.current_stream())
    y = synth.make_inputs(wl, seed=12, device="cuda")
    m2, _ = focus.route(p, y["r"], y["C"])
    q_new.copy_(y["q"][:, -1])
    kc.copy_(y["k"])
    vc.copy_(y["v"])
    mk.copy_(m2)
    graph.replay()
    torch.cuda.synchronize()
    o_ref, l_ref = focus.decode(p, q_new, kc, vc, mk)
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
