"""Device-side failure path without a GPU fault: the attention kernel is run with its
TMA producer held back, so its bounded waits run out (after ~10 ms); it must raise
FOCUS_ERR_TIMEOUT in the status word, abort every role, free its tensor memory and
exit, and the context must stay usable for the next, correct, call."""
import numpy as np
import pytest

import oracle
import synth
from parity import compare_outputs, mask_np

focus = pytest.importorskip("learned_centroid_gated_gb300")

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    assert focus.ERRORS[focus.selftest_timeout()] == "FOCUS_ERR_TIMEOUT"
    assert focus.ERRORS[focus.selftest_timeout()] == "FOCUS_ERR_TIMEOUT"  # twice in a row
    wl = synth.WORKLOADS["tiny"]
    x = synth.make_inputs(wl, seed=6, device="cuda")
    p = focus.Params.from_workload(wl)
    o, lse = focus.attn_fwd(p, x["q"], x["k"], x["v"], x["r"], x["C"])
    ws = focus._default_ws[str(x["q"].device)].buf
    assert focus.get_status(ws) == 0
    mask, _ = focus.route(p, x["r"], x["C"])
    o_ref, lse_ref = oracle.attn(x["q"], x["k"], x["v"], mask_np(mask), w=wl.w)
    compare_outputs(o, lse, o_ref, lse_ref)
