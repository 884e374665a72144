"""Host logic of the multi-GPU path on CPU with two gloo ranks: each rank gets its own
problem (distinct seeded inputs), the job time is the max over ranks and the job
throughput counts every rank's tokens.  The data path has no collective."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = synth.WORKLOADS["tiny"]
        x = synth.make_inputs(wl, seed=bench.rank_seed(0, rank))
        local_ms = 10.0 + 5.0 * rank
        job_ms = bench.reduce_max(local_ms, dist, torch.device("cpu"))
        digest = torch.tensor([float(x["q"].float().sum()), float(x["r"].sum())], dtype=torch.float64)
        gathered = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(gathered, digest)
        out[rank] = (job_ms, [g.tolist() for g in gathered],
                     bench.job_throughput(world, wl.B * wl.N, job_ms / 1e3))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        job_ms, digests, thr = res[rank]
        assert job_ms == pytest.approx(15.0)           # slowest rank
        assert digests[0] != digests[1]                 # independent problems
        assert thr == pytest.approx(2 * 512 / 0.015)    # all ranks' tokens / job time
