"""The debug build (FOCUS_DEBUG_BOUNDS=1: index checks on data-derived indices raise
FOCUS_ERR_BOUNDS on the status word) compiles into its own library with the full C
ABI, and on valid inputs it returns the default build's results, bit for bit, with a
clean status."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BUILD = os.path.join(ROOT, "learned_centroid_gated_gb300", "build.py")
DEBUG_LIB = os.path.join(ROOT, "learned_centroid_gated_gb300", "libfocus_debug.so")


def _build_debug():
    env = dict(os.environ, FOCUS_DEBUG_BOUNDS="1")
    r = subprocess.run([sys.executable, BUILD], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    assert os.path.exists(DEBUG_LIB)


def test_debug_build_exports_the_abi():
    import shutil
    if not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")):
        pytest.skip("nvcc not available")
    _build_debug()
    import re
    header = open(os.path.join(ROOT, "include", "focus.h")).read()
    names = set(re.findall(r"\b(focus_[a-z0-9_]+)\s*\(", header))
    out = subprocess.run(["nm", "-D", "--defined-only", DEBUG_LIB], capture_output=True, text=True).stdout
    missing = sorted(n for n in names if n not in out)
    assert not missing, missing


_CHILD = r"""
import os, sys, json
sys.path.insert(0, sys.argv[1])
import torch
import learned_centroid_gated_gb300 as focus
import synth
wl = synth.WORKLOADS["tiny"].replace(N=1000, H=4, H_kv=2, R=2, d_head=128, K=6, top_k=3, w=100)
x = synth.make_inputs(wl, seed=3, device="cuda")
p = focus.Params.from_workload(wl)
o, lse = focus.attn_fwd(p, x["q"], x["k"], x["v"], x["r"], x["C"])
ws = focus._default_ws[str(x["q"].device)].buf
torch.save({"o": o.cpu(), "lse": lse.cpu(), "status": focus.get_status(ws),
            "lib": os.path.basename(focus.LIB_PATH)}, sys.argv[2])
"""


@pytest.mark.gpu
def test_debug_build_matches_default_build(tmp_path):
    import torch
    _build_debug()
    res = {}
    for tag, env_extra in (("default", {}), ("debug", {"FOCUS_DEBUG_BOUNDS": "1"})):
        env = dict(os.environ, **env_extra)
        env.pop("FOCUS_DEBUG_BOUNDS", None) if tag == "default" else None
        out = str(tmp_path / f"{tag}.pt")
        r = subprocess.run([sys.executable, "-c", _CHILD, ROOT, out], env=env, capture_output=True,
                           text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        res[tag] = torch.load(out)
    assert res["default"]["lib"] == "libfocus.so" and res["debug"]["lib"] == "libfocus_debug.so"
    assert res["default"]["status"] == 0 and res["debug"]["status"] == 0
    assert torch.equal(res["default"]["o"], res["debug"]["o"])
    assert torch.equal(res["default"]["lse"], res["debug"]["lse"])
