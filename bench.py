#!/usr/bin/env python
"""Benchmark of the Focus attention forward pass on GB300; prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl focus|reference]

A step is one full forward pass (routing, bucketing, permuted copies, long-range
and window attention with the union merge) over one synthetic batch whose inputs
are already resident in HBM.  The default workload is the largest one that fits
one GPU: the 1M-token GQA layer (32 query / 8 KV heads, d = 128, K = 4, top_k = 1,
w = 1024).  Timing: W untimed warm-up steps, then K steps between CUDA events on
the launching stream, bracketed by barrier + synchronize, max over ranks; the
median of the per-step durations is reported beside the mean.  Each rank
processes its own independent problem (weak scaling, no collective on the data
path).  The inputs (Q/K/V) are larger than L2, so no flush is needed between
steps.  --tokens N runs the same workload family at N tokens (for profiling).

--impl reference times the CPU oracle (the only comparison implementation: the
pages ship no code) on the host cores, each step a bounded sample of query rows.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "Focus attn fwd tokens/s and allowed-pair TFLOP/s vs GB300 BF16 peak"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "extreme_1m"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 2**20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(synth.WORKLOADS))
    ap.add_argument("--impl", default="focus", choices=["focus", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--tokens", type=int, default=0,
                    help="run the workload family at this many tokens instead (profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--sweep", choices=["table6", "decode", "schedule", "backward", "graph"], default=None,
                    help="table6: speedup of Focus over this build's own dense causal mode "
                         "(K=1) across context lengths, K=4 and K=8; decode: one decode step "
                         "per workload; schedule: exact-set segments vs group lists over "
                         "(K, top_k) at 32K tokens; backward: dq, dk, dv with the masks held "
                         "fixed, per kernel; graph: eager calls vs one captured CUDA graph "
                         "on the launch-bound small layers (one JSON line each)")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            flat = {}
            for k, v in d.items():
                if isinstance(v, (int, float)):
                    flat[k] = float(v)
                elif isinstance(v, dict) and isinstance(v.get("value"), (int, float)):
                    flat[k] = float(v["value"])
            if "bf16_tflops" in flat:
                for k, v in FALLBACK_PEAKS.items():
                    flat.setdefault(k, v)
                return flat, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        sel = []
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            pass
        self.cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "200"] + sel

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        self.out.flush()
        rows = []
        try:
            for line in open(self.out.name):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        except Exception:
            pass
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        reasons = sorted({n for r in rows for n, v in zip(self.NAMES, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "reasons": reasons, "samples": len(rows),
                "power_w_median": statistics.median(float(r[3]) for r in rows
                                                    if r[3].replace(".", "").isdigit())}


def bind_to_gpu_cpus(device_index: int):
    """Restrict this process to the CPU cores NVML names as local to the GPU, so pinned
    host buffers allocated afterwards sit in the memory attached to it: on a box with
    two CPU sockets, buffers on the far socket reach the GPU through the socket link
    (measured 56 GB/s host-to-device against 180-210 from the near one).  Returns the
    core list, or None when NVML cannot say (nothing changes then)."""
    import ctypes
    try:
        nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if nvml.nvmlInit_v2() != 0:
            return None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            h = ctypes.c_void_p()
            if nvml.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
                return None
            n_words = (os.cpu_count() + 63) // 64
            words = (ctypes.c_ulong * n_words)()
            if nvml.nvmlDeviceGetCpuAffinity(h, ctypes.c_uint(n_words), words) != 0:
                return None
            cpus = {64 * i + b for i in range(n_words) for b in range(64) if (words[i] >> b) & 1}
            cpus &= set(range(os.cpu_count()))
            if not cpus:
                return None
            os.sched_setaffinity(0, cpus)
            return sorted(cpus)
        finally:
            nvml.nvmlShutdown()
    except Exception:
        return None


# ------------------------------------------------------------- oracle legs --
def uniform_rows(N: int, n: int, seed: int) -> np.ndarray:
    g = np.random.default_rng(seed)
    return np.sort(g.choice(N, size=min(n, N), replace=False)).astype(np.int64)


def oracle_time_tokens(wl, inputs_cpu, target_s: float, seed: int = 11):
    """Time the CPU oracle on a bounded sample: routing for all N tokens plus the
    attention of a uniform sample of query rows (all heads).  Returns
    (tokens/s, cores, sample description)."""
    import oracle
    cores = oracle.n_cores()
    t0 = time.perf_counter()
    mask, _, _, _ = oracle.route(inputs_cpu["r"], inputs_cpu["C"], K=wl.K, top_k=wl.top_k,
                                 sinkhorn_iters=wl.sinkhorn_iters, sinkhorn_eps=wl.sinkhorn_eps)
    t_route = time.perf_counter() - t0
    q, k, v = inputs_cpu["q"], inputs_cpu["k"], inputs_cpu["v"]
    cal = uniform_rows(wl.N, 8, seed)
    t0 = time.perf_counter()
    oracle.attn(q, k, v, mask, w=wl.w, rows=cal)
    per_row = (time.perf_counter() - t0) / len(cal)
    n = int(max(8, min(wl.N, (target_s - t_route) / max(per_row, 1e-9))))
    rows = uniform_rows(wl.N, n, seed + 1)
    t0 = time.perf_counter()
    oracle.attn(q, k, v, mask, w=wl.w, rows=rows)
    t_attn = time.perf_counter() - t0
    sec_per_token = t_route / wl.N + t_attn / len(rows)
    desc = (f"routing of all {wl.N} tokens ({t_route:.2f} s) + attention of {len(rows)} uniformly "
            f"sampled query rows x {wl.H} heads ({t_attn:.2f} s); tokens/s = 1 / (route s/token + "
            f"attention s/row), batch b=0")
    return 1.0 / sec_per_token, cores, desc, t_route + t_attn


def oracle_single_core_tiny():
    """The oracle on one host core over the whole tiny workload (N = 512, 2 heads):
    routing of every token and attention of every row.  Returns tokens/s."""
    import oracle
    wl = synth.WORKLOADS["tiny"]
    x = synth.make_inputs(wl, seed=0, device="cpu")
    t0 = time.perf_counter()
    mask, _, _, _ = oracle.route(x["r"], x["C"], K=wl.K, top_k=wl.top_k,
                                 sinkhorn_iters=wl.sinkhorn_iters, sinkhorn_eps=wl.sinkhorn_eps)
    oracle.attn(x["q"], x["k"], x["v"], mask, w=wl.w, n_threads=1)
    return wl.B * wl.N / (time.perf_counter() - t0)


def workload_of(args):
    """The bench workload; with --tokens, the same family at that many tokens."""
    wl = synth.WORKLOADS[args.workload]
    if getattr(args, "tokens", 0):
        wl = wl.replace(name=f"{wl.name}_n{args.tokens}", N=args.tokens)
    return wl


def run_reference(args):
    """The oracle on the host cores, on the same workload, metric and config as the
    GPU arm.  Each step is a bounded sample of the workload (routing of every token +
    attention of a uniform sample of query rows, all heads), timed on the host wall
    clock; `value` is the sampled rate in tokens/s and `ms_per_step` the measured
    seconds of one sampled step (not of a whole-workload pass, which is reported,
    extrapolated from the rate, under its own key)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = workload_of(args)
    x = synth.make_inputs(wl, seed=args.seed, device="cpu")
    total = max(1, args.steps + args.warmup)
    per_step = max(2.0, min(10.0, 150.0 / total))
    vals, step_s = [], []
    desc = cores = None
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        v, cores, desc, _ = oracle_time_tokens(wl, x, per_step, seed=100 + i)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            vals.append(v)
            step_s.append(dt)
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * statistics.mean(step_s),
        "ms_per_step_median": 1000.0 * statistics.median(step_s),
        "full_workload_ms_extrapolated": 1000.0 * wl.B * wl.N / value,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step: {desc}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def config_of(wl):
    """The workload description; identical in both arms of the benchmark."""
    return {"workload": wl.name, "B": wl.B, "N": wl.N, "H": wl.H, "H_kv": wl.H_kv,
            "d_head": wl.d_head, "R": wl.R, "K": wl.K, "top_k": wl.top_k, "w": wl.w,
            "sinkhorn_iters": wl.sinkhorn_iters, "softmax_scale": 1.0 / math.sqrt(wl.d_head)}


def group_diagnostics(mask_np: np.ndarray, K: int, top_k: int, margin_np: np.ndarray | None):
    """Group sizes and dominance per (b, routing head), from the masks the kernels
    used, and the near-tie count of the top-k decisions.  Dominance = the largest
    share of tokens that are members of one group (balanced: top_k / K); the pages
    track it as the collapse signal of the grouping (thelatestinai.com list view,
    Table 9; gist.science "Key Technical Innovation: Sinkhorn Normalization")."""
    m = mask_np.astype(np.uint32)
    N = m.shape[-1]
    sizes = np.stack([((m >> g) & 1).sum(axis=-1) for g in range(K)], axis=-1)  # [B, R, K]
    share = sizes / float(N)
    out = {"group_sizes": sizes.tolist(), "dominance": share.max(axis=-1).tolist(),
           "dominance_max": float(share.max()), "balanced_share": top_k / K,
           "smallest_group_share": float(share.min())}
    if margin_np is not None:
        out["near_ties"] = int((margin_np < 1e-5).sum())
        out["near_tie_threshold"] = 1e-5
    return out


def code_hash(path: str) -> str:
    """sha256 of a C/CUDA source with its comments and whitespace removed: a traffic
    capture stays valid across comment edits, not across code changes."""
    src = open(path, encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return hashlib.sha256("".join(src.split()).encode()).hexdigest()


def traffic_of(kernel_src: str, workload: str):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu summary,
    if it was taken on the current kernel source and covers this workload (else
    None).  The file holds one entry per workload; an entry for a workload too large
    to capture under ncu is scaled from captures of the same family at fewer tokens
    (the entry states how)."""
    path = os.path.join(ROOT, "profiles", "attn_long_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
        if d.get("code_sha256") != code_hash(kernel_src):
            return None
        e = d.get("entries", {}).get(workload)
        return None if e is None else e.get("traffic_bytes_per_launch")
    except Exception:
        pass
    return None


def long_range_bytes(wl, group_lists: bool) -> float:
    """Algorithmic DRAM bytes of one long-range launch: the permuted Q', K', V' read
    once (bf16), the window part O_w (fp32) and LSE_w read, O (bf16) and LSE
    written; with group lists the rows are top_k-fold and the list parts (fp32) are
    written instead of O."""
    rep = wl.top_k if group_lists else 1
    qkv = 2.0 * wl.B * wl.N * rep * (wl.H + 2 * wl.H_kv) * wl.d_head
    rows = wl.B * wl.N * wl.H
    if group_lists:
        return qkv + rows * rep * (4.0 * wl.d_head + 4.0)
    return qkv + rows * (4.0 * wl.d_head + 4.0) + rows * (2.0 * wl.d_head + 4.0)


# ------------------------------------------------------------ multi-rank --
def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank processes its own independent problem (weak scaling)."""
    return base_seed + rank


def reduce_max(value: float, dist, device) -> float:
    """Max of a per-rank scalar over all ranks (the job's time is its slowest rank)."""
    if dist is None:
        return value
    t = torch.tensor([value], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, units_per_rank: float, seconds: float) -> float:
    """Whole-job units per second: every rank processed units_per_rank in <= seconds."""
    return world * units_per_rank / seconds


# ---------------------------------------------------------------- GPU arm --
def run_focus(args):
    import learned_centroid_gated_gb300 as focus
    from learned_centroid_gated_gb300 import pairs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    affinity = bind_to_gpu_cpus(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    wl = workload_of(args)
    p = focus.Params.from_workload(wl)
    x = synth.make_inputs(wl, seed=rank_seed(args.seed, rank), device=dev)
    ws = focus.Workspace(dev).get(p)
    o = torch.empty_like(x["q"])
    lse = torch.empty(p.B, p.H, p.N, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        focus.attn_fwd(p, x["q"], x["k"], x["v"], x["r"], x["C"], out=o, lse=lse, ws=ws,
                       stream=stream, stage_events=evs)

    W, K = max(args.warmup, 3), args.steps
    for _ in range(W):
        step()
    torch.cuda.synchronize()
    status = focus.get_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {status}: {focus.strerror(status)}")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(focus.N_STAGE_EVENTS)]
           for _ in range(K)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        time.sleep(0.3)
        step()  # the clocks ramp under load before the timed region
        barrier()
        t_start.record(stream)
        for i in range(K):
            step(evs[i])
        t_end.record(stream)
        barrier()
        time.sleep(0.1)
    clocks = clk.summary()
    ms = reduce_max(t_start.elapsed_time(t_end), dist, dev)
    ms_step = ms / K
    step_ms = [e[0].elapsed_time(e[-1]) for e in evs]
    ms_median = reduce_max(statistics.median(step_ms), dist, dev)
    stage_ms = {}
    for si, name in enumerate(focus.STAGES):
        stage_ms[name] = statistics.mean(e[si].elapsed_time(e[si + 1]) for e in evs)

    value = job_throughput(world, wl.B * wl.N, ms_step / 1e3)

    # exact allowed-pair accounting from the membership the kernels used
    mask, margin = focus.route(p, x["r"], x["C"], margin=True)
    mask_np = mask.cpu().numpy().view(np.uint32)
    margin_np = margin.cpu().numpy()
    cnt = pairs.allowed_pairs(mask_np, wl.w)  # [B, R]
    heads_per_rho = wl.H // wl.R
    allowed = int(cnt.sum()) * heads_per_rho
    window = pairs.window_pairs(wl.N, wl.w) * wl.B * wl.H
    longrange = allowed - window
    flops = 4.0 * wl.d_head * allowed
    flops_long = 4.0 * wl.d_head * longrange
    tflops = flops / (ms_step / 1e3) / 1e12
    # executed tensor-core work (whole 256 x 128 tiles, masked elements included)
    group_lists = p.bucket_shape()[0] == focus.SCHEDULE_GROUPS
    lt, wt = pairs.executed_tiles(mask_np, wl.w, group_lists=group_lists)
    tile_flops = 4.0 * wl.d_head * 256 * 128
    exec_long = tile_flops * int(lt.sum()) * heads_per_rho
    exec_win = tile_flops * wt * wl.B * wl.H
    causal = wl.B * wl.H * wl.N * (wl.N + 1) // 2

    # end-to-end through the public host-buffer API (pinned host inputs, filled by DMA
    # from the device copies so both legs see the same data); the host entry holds its
    # own workspace, the device-resident one stays for the interleaved steps below
    host = {}
    for n, t in x.items():
        host[n] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        host[n].copy_(t)
    torch.cuda.synchronize()
    # raw copy rates of these pinned buffers (one flat copy of Q each way)
    xq = torch.empty_like(x["q"])
    c0, c1, c2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    c0.record(stream)
    xq.copy_(host["q"], non_blocking=True)
    c1.record(stream)
    host["q"].copy_(xq, non_blocking=True)
    c2.record(stream)
    c2.synchronize()
    qb = xq.numel() * xq.element_size()
    copy_rates = {"h2d_gbs": qb / c0.elapsed_time(c1) / 1e6, "d2h_gbs": qb / c1.elapsed_time(c2) / 1e6}
    del xq
    # After a long device-timed region (the 1M-token layer runs ~40 s at the power
    # cap) the GPU is hotter than when that region started and holds lower clocks for
    # the same power; an idle pause lets the end-to-end leg start from a comparable
    # state (each call was measured drifting from 1.70 to 2.06 s over a minute of load)
    cooldown = 15.0 if ms_step * (K + W) / 1e3 > 10.0 else 0.0
    time.sleep(cooldown)
    sess = focus.HostSession(p, dev)
    for _ in range(3):
        sess(host["q"], host["k"], host["v"], host["r"], host["C"])
    barrier()
    ke = max(3, min(K, 10))
    e_times, d_times = [], []
    with ClockSampler(local) as eclk:
        for _ in range(ke):
            # one device-resident step right before each call: the same box, clocks and
            # thermal state as the call, for the ratio below
            d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            d0.record(stream)
            step()
            d1.record(stream)
            d1.synchronize()
            d_times.append(d0.elapsed_time(d1))
            e0 = time.perf_counter()  # each call returns after its outputs are on the host
            sess(host["q"], host["k"], host["v"], host["r"], host["C"])
            e_times.append(time.perf_counter() - e0)
        barrier()
    e_clocks = eclk.summary()
    del ws, o, lse
    # median of the calls' wall times (a single slow call of the host process would
    # otherwise dominate a mean of a few calls); the mean is reported beside it
    e_s = reduce_max(statistics.median(e_times), dist, dev)
    e2e = {"value": job_throughput(world, wl.B * wl.N, e_s), "unit": UNIT,
           "h2d_bytes_per_step": sess.h2d_bytes(*host.values()),
           "d2h_bytes_per_step": sess.d2h_bytes(), "ms_per_step": 1e3 * e_s,
           "ms_per_step_mean": 1e3 * statistics.mean(e_times), "calls": ke,
           "call_ms": [round(1e3 * t, 2) for t in e_times],
           "over_device_ms": e_s * 1e3 / ms_step,
           "device_ms_interleaved": statistics.median(d_times),
           "over_device_interleaved": e_s * 1e3 / statistics.median(d_times),
           "copy_rates": copy_rates,
           "cpu_affinity": (f"{len(affinity)} GPU-local cores (NVML)" if affinity else "unchanged"),
           "head_groups": sess.group_sizes(), "cooldown_s": cooldown, "clocks": e_clocks}
    del host, sess

    peaks, peak_src = load_peaks()
    t_long = stage_ms["attn_long"] / 1e3
    achieved = flops_long / t_long / 1e12
    sched = "kGrp" if group_lists else "kSeg"
    roofline = {
        "kernel": f"attn_tc<{wl.d_head}, {sched}> (long-range block-sparse attention, tcgen05)",
        "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
        "frac": achieved / peaks["bf16_tflops"],
        "peak_source": f"{peak_src} bf16 dense burst",
        "peak_sustained": peaks["bf16_tflops_sustained"],
        "frac_sustained": achieved / peaks["bf16_tflops_sustained"],
        "traffic": traffic_of(
            os.path.join(ROOT, "learned_centroid_gated_gb300", "csrc", "attn_tc.cu"), wl.name),
        "algorithmic_bytes_per_launch": long_range_bytes(wl, group_lists),
        "algorithmic_flops_per_launch": flops_long,
        "executed_flops_per_launch": exec_long,
        "tile_efficiency": flops_long / exec_long,
        "executed_tflops": exec_long / t_long / 1e12,
        "launch_ms": stage_ms["attn_long"],
    }
    # route (+ 2 per Sinkhorn iteration), 3 bucketing, schedule, plan, permute,
    # window, long-range (+ the slot merge under group lists)
    launches_per_step = (1 + 2 * wl.sinkhorn_iters) + 3 + 1 + 1 + 1 + 1 + 1 \
        + (1 if group_lists else 0)
    qkv_bytes = sum(x[n].numel() * x[n].element_size() for n in ("q", "k", "v"))

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_step, "ms_per_step_median": ms_median,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": config_of(wl),
        "l2": f"inputs larger than L2 (Q/K/V {qkv_bytes / 2**20:.0f} MiB > {L2_BYTES / 2**20:.0f} MiB), "
              "no flush",
        "parallelism": f"independent problem per GPU x{world}",
        "schedule": "groups" if group_lists else "segments",
        "allowed_pair_tflops": tflops,
        "allowed_pair_frac_of_peak": tflops / peaks["bf16_tflops"],
        "allowed_pairs": allowed, "allowed_fraction_of_causal": allowed / causal,
        "stages_ms": stage_ms,
        "window": {"algorithmic_tflops": 4.0 * wl.d_head * window / (stage_ms["attn_window"] / 1e3) / 1e12,
                   "executed_tflops": exec_win / (stage_ms["attn_window"] / 1e3) / 1e12,
                   "tile_efficiency": 4.0 * wl.d_head * window / exec_win},
        "groups": group_diagnostics(mask_np, wl.K, wl.top_k, margin_np),
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        xc = {n: t.cpu() for n, t in x.items()}
        v, cores, desc, secs = oracle_time_tokens(wl, xc, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": desc, "seconds": secs,
                                "single_core_tiny": {"value": oracle_single_core_tiny(), "unit": UNIT,
                                                     "cores": 1, "sample": "whole tiny workload "
                                                     "(N=512, 2 heads, d=64): routing + every row"}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------------- Table 6 --
# "Why Attend to Everything? Focus is the Key", thelatestinai.com list view,
# Table 6: wall-clock speedup of Focus over full attention (both FlashAttention) on
# H100-80GB at 1K..1M tokens, K=4 and K=8.  The pages do not state the model, head
# count, head size, top_k or window; the sweep below uses 32 query / 8 KV heads,
# d=128, top_k=1, w=1024 and compares with this build's own dense causal mode
# (K=1: every key is in the single group, so the long-range part is all causal keys).
TABLE6_PAGES = {"context": [1024, 4096, 16384, 32768, 65536, 262144, 1048576],
                "K4": [0.2, 0.5, 1.5, 2.2, 3.0, 4.0, 4.1], "K8": [0.2, 0.6, 1.8, 3.1, 4.7, 7.6, 8.6]}


def run_table6(args):
    import learned_centroid_gated_gb300 as focus
    from learned_centroid_gated_gb300 import pairs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    base = synth.Workload("table6", B=1, N=1024, H=32, H_kv=8, d_head=128, R=1, K=1, top_k=1, w=1024)
    rows = []
    for N in TABLE6_PAGES["context"]:
        wl0 = base.replace(N=N)
        x = synth.make_qkv(wl0, seed=args.seed, device=dev)
        ws = focus.Workspace(dev)
        o = torch.empty_like(x[0])
        res = {"N": N}
        for tag, K in (("dense", 1), ("K4", 4), ("K8", 8)):
            wl = wl0.replace(K=K)
            r, C = synth.make_routing(wl, seed=args.seed, device=dev)
            p = focus.Params.from_workload(wl)
            steps = 2 if N >= 262144 else 5
            for _ in range(2):
                focus.attn_fwd(p, *x, r, C, out=o, want_lse=False, ws=ws, stream=stream)
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            t0.record(stream)
            for _ in range(steps):
                focus.attn_fwd(p, *x, r, C, out=o, want_lse=False, ws=ws, stream=stream)
            t1.record(stream)
            torch.cuda.synchronize()
            ms = t0.elapsed_time(t1) / steps
            mask, _ = focus.route(p, r, C, ws=ws)
            allowed = int(pairs.allowed_pairs(mask.cpu().numpy().view(np.uint32), wl.w).sum()) * wl.H
            res[f"{tag}_ms"] = ms
            res[f"{tag}_allowed_pair_tflops"] = 4.0 * wl.d_head * allowed / (ms / 1e3) / 1e12
            res[f"{tag}_pairs_retained"] = allowed / (wl.H * N * (N + 1) // 2)
        res["speedup_K4"] = res["dense_ms"] / res["K4_ms"]
        res["speedup_K8"] = res["dense_ms"] / res["K8_ms"]
        rows.append(res)
        del x, ws, o
        torch.cuda.empty_cache()
    print(json.dumps({"sweep": "table6", "unit": "ms per forward", "dtype": "bf16", "data": "synthetic",
                      "config": {"B": 1, "H": 32, "H_kv": 8, "d_head": 128, "R": 1, "top_k": 1,
                                 "w": 1024, "dense": "K=1 (all causal keys)"},
                      "rows": rows, "pages_table6_h100": TABLE6_PAGES}), flush=True)


# -------------------------------------------------------------- decode --
def run_decode(args):
    """Decode step (newest token over its cache) per workload: time, tokens/s and
    the HBM roofline (algorithmic bytes = the allowed keys' K and V rows of every KV
    head + the masks + q and o)."""
    import learned_centroid_gated_gb300 as focus

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()
    rows = []
    for name in ("mha7b_32k", "gqa_128k", "extreme_1m"):
        wl = synth.WORKLOADS[name]
        x = synth.make_inputs(wl, seed=args.seed, device=dev)
        p = focus.Params.from_workload(wl)
        mask, _ = focus.route(p, x["r"], x["C"])
        q_new = x["q"][:, wl.N - 1].contiguous()
        m = mask.cpu().numpy().view(np.uint32)
        allowed_keys = 0
        for b in range(wl.B):
            for rho in range(wl.R):
                mm = m[b, rho]
                i = wl.N - 1
                j = np.arange(wl.N)
                ok = (i - j < wl.w) | ((mm & mm[i]) != 0)
                allowed_keys += int(ok.sum()) * (wl.H_kv // wl.R)
        byts = allowed_keys * 2 * wl.d_head * 2 + wl.B * wl.R * wl.N * 4 + 2 * wl.B * wl.H * wl.d_head * 2
        ws = torch.empty(focus.decode_workspace_size(p), dtype=torch.uint8, device=dev)
        o = torch.empty(wl.B, wl.H, wl.d_head, dtype=torch.bfloat16, device=dev)
        for _ in range(5):
            focus.decode(p, q_new, x["k"], x["v"], mask, out=o, want_lse=False, ws=ws, stream=stream)
        # > L2, read between steps: the cache then holds clean lines of another buffer
        # (a write-based flush would leave dirty lines whose write-back lands in the step)
        flush = torch.zeros(64 * 2**20, dtype=torch.float32, device=dev)
        times = []
        for _ in range(20):
            flush.max()
            # keep the device busy while the host enqueues the step, so that the events
            # time the step's kernels rather than the Python call
            torch.cuda._sleep(200_000)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            focus.decode(p, q_new, x["k"], x["v"], mask, out=o, want_lse=False, ws=ws, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        gbs = byts / (ms / 1e3) / 1e9
        rows.append({"workload": name, "ms": ms, "tokens_per_s": wl.B / (ms / 1e3),
                     "algorithmic_bytes": byts, "achieved_gbs": gbs, "hbm_frac": gbs / peaks["hbm_gbs"],
                     "allowed_key_fraction": allowed_keys / (wl.B * wl.H_kv * wl.N)})
        del x, ws, flush
        torch.cuda.empty_cache()
    print(json.dumps({"sweep": "decode", "unit": "ms per decode step",
                      "l2": "flushed before each step (a 256 MiB read)",
                      "timing": "device time of the step's kernels (host enqueue hidden)",
                      "peak_hbm_gbs": peaks["hbm_gbs"], "peak_source": peak_src, "rows": rows}), flush=True)


# ------------------------------------------------------------ schedules --
SCHEDULE_GRID = [(4, 2, 32768), (8, 2, 32768), (8, 4, 32768), (16, 2, 32768), (32, 2, 32768),
                 (16, 4, 32768), (32, 4, 32768), (8, 2, 131072), (16, 2, 131072)]


def run_schedule(args):
    """Exact-set segments vs group lists on a 32-head, d=128 layer (w=512) for
    several (K, top_k, N): step time, its stages, and allowed-pair TFLOP/s.  Segments
    run only while C(K, top_k) <= 1024."""
    import math

    import learned_centroid_gated_gb300 as focus
    from learned_centroid_gated_gb300 import pairs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    base = synth.WORKLOADS["mha7b_32k"]
    rows = []
    x, o = None, None
    for K, top_k, N in SCHEDULE_GRID:
        wl = base.replace(K=K, top_k=top_k, N=N)
        if x is None or x[0].shape[1] != N:
            x = o = None
            torch.cuda.empty_cache()
            x = synth.make_qkv(wl, seed=args.seed, device=dev)
            o = torch.empty_like(x[0])
        r, C = synth.make_routing(wl, seed=args.seed, device=dev)
        p0 = focus.Params.from_workload(wl)
        mask, _ = focus.route(p0, r, C)
        allowed = int(pairs.allowed_pairs(mask.cpu().numpy().view(np.uint32), wl.w).sum()) * wl.H
        flops = 4.0 * wl.d_head * allowed
        for sch in (focus.SCHEDULE_SEGMENTS, focus.SCHEDULE_GROUPS):
            if sch == focus.SCHEDULE_SEGMENTS and math.comb(K, top_k) > 1024:
                continue
            p = focus.Params.from_workload(wl, schedule=sch)
            ws = focus.Workspace(dev).get(p)
            for _ in range(3):
                focus.attn_fwd(p, *x, r, C, out=o, want_lse=False, ws=ws, stream=stream)
            torch.cuda.synchronize()
            assert focus.get_status(ws) == 0
            steps = 5
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(focus.N_STAGE_EVENTS)]
                   for _ in range(steps)]
            for e in evs:
                focus.attn_fwd(p, *x, r, C, out=o, want_lse=False, ws=ws, stream=stream,
                               stage_events=e)
            torch.cuda.synchronize()
            stage = {n: statistics.median(e[i].elapsed_time(e[i + 1]) for e in evs)
                     for i, n in enumerate(focus.STAGES)}
            ms = statistics.median(e[0].elapsed_time(e[-1]) for e in evs)
            rows.append({"K": K, "top_k": top_k, "N": N, "sets": math.comb(K, top_k),
                         "schedule": "segments" if sch == focus.SCHEDULE_SEGMENTS else "groups",
                         "auto": p0.bucket_shape()[0] == sch, "ms": ms,
                         "tokens_per_s": wl.B * wl.N / (ms / 1e3),
                         "allowed_pair_tflops": flops / (ms / 1e3) / 1e12,
                         "pairs_retained": allowed / (wl.H * wl.N * (wl.N + 1) // 2),
                         "stages_ms": stage})
            del ws
            torch.cuda.empty_cache()
    print(json.dumps({"sweep": "schedule", "unit": "ms per forward", "dtype": "bf16",
                      "data": "synthetic",
                      "config": config_of(base) | {"K": "varies", "top_k": "varies", "N": "varies"},
                      "note": "attn_long includes the slot merge under group lists",
                      "rows": rows}), flush=True)


# ------------------------------------------------------------- backward --
def run_backward(args):
    """Backward pass (hard mask held fixed) per workload: the forward for reference,
    the backward's stages, and tensor-core rates.  Work is counted on allowed pairs:
    the forward's 2 products (4 d flops per pair), the backward's 5 (10 d: S, dP, dQ,
    dK, dV); its kernels execute 7 (dQ recomputes S and dP: the long-range dQ kernel
    runs 3 products, the dK/dV kernel 4)."""
    import learned_centroid_gated_gb300 as focus
    from learned_centroid_gated_gb300 import pairs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()
    rows = []
    cases = [("mha7b_32k", synth.WORKLOADS["mha7b_32k"]), ("gqa_128k", synth.WORKLOADS["gqa_128k"]),
             ("mha7b_32k_K32_top4", synth.WORKLOADS["mha7b_32k"].replace(K=32, top_k=4))]
    for name, wl in cases:
        x = synth.make_inputs(wl, seed=args.seed, device=dev)
        p = focus.Params.from_workload(wl)
        mask, _ = focus.route(p, x["r"], x["C"])
        o, lse = focus.attn_fwd(p, x["q"], x["k"], x["v"], mask=mask)
        g = torch.Generator(device="cpu").manual_seed(args.seed + 1)
        d_o = torch.randn(x["q"].shape, generator=g).to(torch.bfloat16).to(dev)
        ws = torch.empty(focus.bwd_workspace_size(p), dtype=torch.uint8, device=dev)
        grads = (torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"]))
        run = lambda evs=None: focus.attn_bwd(p, x["q"], x["k"], x["v"], mask, o, lse, d_o, dq=grads[0],
                                             dk=grads[1], dv=grads[2], ws=ws, stream=stream, stage_events=evs)
        for _ in range(max(args.warmup, 2)):
            run()
        torch.cuda.synchronize()
        status = focus.get_status(ws)
        if status != 0:
            raise RuntimeError(f"device status {status}")
        steps = 5
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(focus.N_BWD_STAGE_EVENTS)]
               for _ in range(steps)]
        for e in evs:
            run(e)
        torch.cuda.synchronize()
        stage = {n: statistics.median(e[i].elapsed_time(e[i + 1]) for e in evs)
                 for i, n in enumerate(focus.BWD_STAGES)}
        bwd_ms = statistics.median(e[0].elapsed_time(e[-1]) for e in evs)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(steps):
            focus.attn_fwd(p, x["q"], x["k"], x["v"], mask=mask, out=o, lse=lse, stream=stream)
        f1.record(stream)
        torch.cuda.synchronize()
        fwd_ms = f0.elapsed_time(f1) / steps
        allowed = int(pairs.allowed_pairs(mask.cpu().numpy().view(np.uint32), wl.w).sum()) * (wl.H // wl.R)
        window = pairs.window_pairs(wl.N, wl.w) * wl.B * wl.H
        longr = allowed - window
        d = wl.d_head
        tf = lambda flops, ms: flops / (ms / 1e3) / 1e12
        dkdv = tf(8.0 * d * longr, stage["long_dkdv"])
        rows.append({
            "workload": name, "config": config_of(wl),
            "schedule": "groups" if p.bucket_shape()[0] == focus.SCHEDULE_GROUPS else "segments",
            "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
            "bwd_over_fwd": bwd_ms / fwd_ms, "stages_ms": stage,
            "fwd_allowed_pair_tflops": tf(4.0 * d * allowed, fwd_ms),
            "bwd_allowed_pair_tflops": tf(10.0 * d * allowed, bwd_ms),
            "bwd_executed_tflops": tf(14.0 * d * allowed, bwd_ms),
            "long_dq_tflops": tf(6.0 * d * longr, stage["long_dq"]),
            "long_dkdv_tflops": dkdv,
            "roofline": {"kernel": "bwd_dkdv (long range, tcgen05)", "bound": "tensor",
                         "achieved": dkdv, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": dkdv / peaks["bf16_tflops"], "peak_source": peak_src},
        })
        del x, ws, o, lse, d_o, grads
        torch.cuda.empty_cache()
    print(json.dumps({"sweep": "backward", "unit": "ms per pass", "dtype": "bf16", "data": "synthetic",
                      "l2": "inputs larger than L2, no flush", "rows": rows}), flush=True)


# ---------------------------------------------------------------- graph --
def run_graph(args):
    """Forward pass on the small layers (launch-bound: nine launches per call), eager
    against the replay of one captured CUDA graph, same buffers, CUDA events."""
    import learned_centroid_gated_gb300 as focus

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    rows = []
    for name in ("tiny", "gpt2_layer"):
        wl = synth.WORKLOADS[name]
        p = focus.Params.from_workload(wl)
        x = synth.make_inputs(wl, seed=args.seed, device=dev)
        ws = focus.Workspace(dev).get(p)
        o = torch.empty_like(x["q"])
        lse = torch.empty(p.B, p.H, p.N, dtype=torch.float32, device=dev)
        side = torch.cuda.Stream(dev)
        call = lambda st: focus.attn_fwd(p, x["q"], x["k"], x["v"], x["r"], x["C"], out=o, lse=lse,
                                         ws=ws, stream=st)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for _ in range(3):
                call(side)
        torch.cuda.current_stream(dev).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call(torch.cuda.current_stream(dev))
        stream = torch.cuda.current_stream(dev)
        steps = 200

        def timed(fn):
            for _ in range(10):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / steps

        eager = timed(lambda: call(stream))
        replay = timed(graph.replay)
        rows.append({"workload": name, "config": config_of(wl),
                     "schedule": "groups" if p.bucket_shape()[0] == focus.SCHEDULE_GROUPS else "segments",
                     "eager_ms": eager, "graph_ms": replay,
                     "eager_tokens_per_s": wl.B * wl.N / (eager / 1e3),
                     "graph_tokens_per_s": wl.B * wl.N / (replay / 1e3)})
    print(json.dumps({"sweep": "graph", "unit": "ms per forward", "dtype": "bf16", "data": "synthetic",
                      "rows": rows}), flush=True)


def main():
    args = parse_args()
    if args.sweep == "graph":
        run_graph(args)
        return
    if args.sweep == "backward":
        run_backward(args)
        return
    if args.sweep == "schedule":
        run_schedule(args)
        return
    if args.sweep == "table6":
        run_table6(args)
        return
    if args.sweep == "decode":
        run_decode(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_focus(args)


if __name__ == "__main__":
    main()
