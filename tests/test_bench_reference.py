"""The benchmark's reference arm on the host cores (no GPU): one JSON line with the
contract's keys, the oracle as the comparison implementation; ranks other than 0
print nothing and exit 0."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra):
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [ln for ln in r.stdout.splitlines() if ln.strip()]


def test_reference_arm_prints_one_contract_line():
    lines = _run({})
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["data"] == "synthetic" and d["config"]["workload"] == "tiny"
    assert d["ms_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["gpu_launches"] == 0


def test_reference_arm_other_ranks_stay_silent():
    assert _run({"RANK": "1"}) == []


def test_cpu_binding_never_raises_without_nvml_or_gpu():
    """bench.bind_to_gpu_cpus asks NVML for the GPU-local cores; where NVML or the GPU is
    missing it must leave the affinity alone and return None, not fail the bench."""
    sys.path.insert(0, ROOT)
    import bench
    before = os.sched_getaffinity(0)
    res = bench.bind_to_gpu_cpus(0)
    assert res is None or (isinstance(res, list) and res)
    if res is None:
        assert os.sched_getaffinity(0) == before
    else:
        os.sched_setaffinity(0, before)


def test_code_hash_ignores_comments_not_code(tmp_path):
    """The traffic capture stays valid across comment and whitespace edits of the
    kernel source and is voided by a code change."""
    sys.path.insert(0, ROOT)
    import bench
    a = tmp_path / "a.cu"
    a.write_text("int f(int x) {  // one\n  return x + 1; /* two */\n}\n")
    b = tmp_path / "b.cu"
    b.write_text("// header\nint f(int x)\n{\n  return x + 1;\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) { return x + 2; }\n")
    assert bench.code_hash(str(a)) == bench.code_hash(str(b))
    assert bench.code_hash(str(a)) != bench.code_hash(str(c))
