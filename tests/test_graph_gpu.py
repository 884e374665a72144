"""The forward and backward passes capture into CUDA graphs (GPU).

Small layers are launch-bound (nine launches per forward), so a serving loop
replays one captured graph instead.  Every call enqueues only stream work on the
caller's stream (the tensor maps and kernel attributes are set on the host), so
capture is legal; a replay on new inputs copied into the captured buffers must
equal the eager call bit for bit."""
import pytest
import torch

import synth

focus = pytest.importorskip("learned_centroid_gated_gb300")

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("schedule", [focus.SCHEDULE_SEGMENTS, focus.SCHEDULE_GROUPS])
def test_forward_graph_replay_equals_eager(schedule):
    wl = synth.WORKLOADS["gpt2_layer"]
    p = focus.Params.from_workload(wl, schedule=schedule)
    static = synth.make_inputs(wl, seed=1, device="cuda")
    ws = focus.Workspace("cuda").get(p)
    o = torch.empty_like(static["q"])
    lse = torch.empty(p.B, p.H, p.N, dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm up (tensor maps, attributes) outside capture
        focus.attn_fwd(p, static["q"], static["k"], static["v"], static["r"], static["C"], out=o,
                       lse=lse, ws=ws, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        focus.attn_fwd(p, static["q"], static["k"], static["v"], static["r"], static["C"], out=o,
                       lse=lse, ws=ws, stream=torch.cuda.current_stream())
    for seed in (2, 3):
        fresh = synth.make_inputs(wl, seed=seed, device="cuda")
        for name, t in fresh.items():
            static[name].copy_(t)
        graph.replay()
        torch.cuda.synchronize()
        assert focus.get_status(ws) == 0
        o_ref, l_ref = focus.attn_fwd(p, fresh["q"], fresh["k"], fresh["v"], fresh["r"], fresh["C"])
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_backward_graph_replay_equals_eager():
    wl = synth.WORKLOADS["gpt2_layer"]
    p = focus.Params.from_workload(wl)
    x = synth.make_inputs(wl, seed=4, device="cuda")
    mask, _ = focus.route(p, x["r"], x["C"])
    o, lse = focus.attn_fwd(p, x["q"], x["k"], x["v"], mask=mask)
    d_o = torch.randn_like(x["q"])
    ws = torch.empty(focus.bwd_workspace_size(p), dtype=torch.uint8, device="cuda")
    grads = (torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"]))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        focus.attn_bwd(p, x["q"], x["k"], x["v"], mask, o, lse, d_o, dq=grads[0], dk=grads[1],
                       dv=grads[2], ws=ws, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        focus.attn_bwd(p, x["q"], x["k"], x["v"], mask, o, lse, d_o, dq=grads[0], dk=grads[1],
                       dv=grads[2], ws=ws, stream=torch.cuda.current_stream())
    d_o.copy_(torch.randn_like(d_o))
    graph.replay()
    torch.cuda.synchronize()
    ref = focus.attn_bwd(p, x["q"], x["k"], x["v"], mask, o, lse, d_o)
    for g, r in zip(grads, ref):
        assert torch.equal(g, r)
