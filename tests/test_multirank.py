"""Host logic of the multi-GPU path on CPU with two gloo ranks.

1. Weak scaling as the benchmark runs it: each rank gets its own problem (distinct
   seeded inputs), the job time is the max over ranks and the job throughput
   counts every rank's tokens.  The data path has no collective.
2. One problem sharded over the ranks with no exchange (the partition module):
   every (batch row, query head) is owned by exactly one rank, each rank's routing
   heads are the ones its KV heads read, and the oracle run on each rank's slice
   alone reproduces the unsharded oracle's outputs for those heads bit for bit
   (so no data from another rank is needed)."""
import itertools
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
import synth
from learned_centroid_gated_gb300 import partition


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


@pytest.mark.parametrize("B,H,H_kv,R", [(1, 32, 8, 8), (1, 32, 8, 1), (1, 32, 32, 1), (2, 32, 8, 8),
                                        (3, 32, 8, 2), (4, 4, 1, 1)])
@pytest.mark.parametrize("world", [1, 2, 4, 8])
def test_partition_covers_every_head_once(B, H, H_kv, R, world):
    gq, kv_per_rho = H // H_kv, H_kv // R
    owner = {}
    for rank in range(world):
        s = partition.shard(B, H, H_kv, R, world, rank)
        if s.empty:
            continue
        for b, h in itertools.product(range(s.b0, s.b1), range(s.h0, s.h1)):
            assert (b, h) not in owner, (b, h)
            owner[(b, h)] = rank
            kvh = h // gq
            assert s.kv0 <= kvh < s.kv1                          # its KV head is local
            assert s.rho0 <= kvh // kv_per_rho < s.rho1          # and its routing head
        if R > 1:
            assert s.kv0 % kv_per_rho == 0 and s.kv1 % kv_per_rho == 0   # whole routing heads
    assert len(owner) == B * H


def _shard_worker(rank, world, port, case, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = synth.WORKLOADS["tiny"].replace(**case)
        x = synth.make_inputs(wl, seed=3)                  # every rank sees the same problem
        s = partition.shard(wl.B, wl.H, wl.H_kv, wl.R, world, rank)
        xs = partition.slice_inputs(x, s)
        sub = wl.replace(B=s.b1 - s.b0, H=s.h1 - s.h0, H_kv=s.kv1 - s.kv0, R=s.rho1 - s.rho0)
        mask, _, _, _ = oracle.route(xs["r"], xs["C"], K=sub.K, top_k=sub.top_k)
        o, lse = oracle.attn(xs["q"], xs["k"], xs["v"], mask, w=sub.w, n_threads=2)
        out[rank] = (s, o.reshape(sub.B, sub.N, sub.H, sub.d_head), lse.reshape(sub.B, sub.N, sub.H))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", [dict(B=1, N=300, H=8, H_kv=4, R=2, K=5, top_k=2, w=40),
                                  dict(B=2, N=260, H=4, H_kv=1, R=1, K=4, top_k=2, w=30),
                                  dict(B=1, N=257, H=6, H_kv=2, R=1, K=3, top_k=1, w=17)])
def test_sharded_oracle_equals_unsharded(case):
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_shard_worker, args=(world, port, case, out), nprocs=world, join=True)
        res = dict(out)
    wl = synth.WORKLOADS["tiny"].replace(**case)
    x = synth.make_inputs(wl, seed=3)
    mask, _, _, _ = oracle.route(x["r"], x["C"], K=wl.K, top_k=wl.top_k)
    o, lse = oracle.attn(x["q"], x["k"], x["v"], mask, w=wl.w)
    o = o.reshape(wl.B, wl.N, wl.H, wl.d_head)
    lse = lse.reshape(wl.B, wl.N, wl.H)
    seen = np.zeros((wl.B, wl.H), bool)
    for rank in range(world):
        s, o_r, l_r = res[rank]
        if s.empty:
            continue
        np.testing.assert_array_equal(o_r, o[s.b0:s.b1, :, s.h0:s.h1])
        np.testing.assert_array_equal(l_r, lse[s.b0:s.b1, :, s.h0:s.h1])
        seen[s.b0:s.b1, s.h0:s.h1] = True
    assert seen.all()
