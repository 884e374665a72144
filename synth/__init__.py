"""Seeded synthetic inputs for Focus centroid-gated attention.

This module is shared by the CUDA path's tests/benchmark and by the CPU oracle's
tests. It holds none of the method's arithmetic: it only draws tensors with the
shapes and value distributions of the workloads, and the workload table itself.

Workloads (shapes and distributions as the Focus problem is stated; routing
dimension d_g = 16 from "Why Attend to Everything? Focus is the Key", gist.science
technical summary, section 2 "Core Architecture", and the jindou-blog deep read,
method bullets):

* ``tiny``        B=1 H=2 d=64 N=512, K=4 top_k=2 w=64, no Sinkhorn.
* ``gpt2_layer``  B=1 H=12 d=64 N=4096, r = x W_r with x ~ N(0, I_768) and
                  W_r ~ N(0, 1/768) (768 -> 16); K=4 top_k=2 w=256; 3 Sinkhorn
                  iterations.
* ``mha7b_32k``   B=1 H=32 d=128 N=32768, K=4 top_k=2 w=512.
* ``gqa_128k``    B=1 H=32 H_kv=8 d=128 N=131072, one routing vector per KV-head
                  group (R=8), K=8 top_k=2 w=1024.
* ``extreme_1m``  B=1 H=32 H_kv=8 d=128 N=1048576, K=4 top_k=1 w=1024.

Q, K, V are iid N(0,1) rounded to bf16; routing vectors r are fp32 (iid N(0, I_16)
unless stated); centroids C are fp32 iid N(0,1). The pages evaluate on PG-19 text
with pretrained weights; these seeded draws stand in for that data.
"""
from __future__ import annotations

import dataclasses
import math

import torch

D_G = 16  # routing dimension


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    N: int
    H: int
    H_kv: int
    d_head: int
    R: int
    K: int
    top_k: int
    w: int
    sinkhorn_iters: int = 0
    sinkhorn_eps: float = 1.0
    routing: str = "iid"  # "iid" or "proj768"

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d_head)


WORKLOADS = {
    "tiny": Workload("tiny", B=1, N=512, H=2, H_kv=2, d_head=64, R=1, K=4, top_k=2, w=64),
    "gpt2_layer": Workload("gpt2_layer", B=1, N=4096, H=12, H_kv=12, d_head=64, R=1, K=4,
                           top_k=2, w=256, sinkhorn_iters=3, routing="proj768"),
    "mha7b_32k": Workload("mha7b_32k", B=1, N=32768, H=32, H_kv=32, d_head=128, R=1, K=4,
                          top_k=2, w=512),
    "gqa_128k": Workload("gqa_128k", B=1, N=131072, H=32, H_kv=8, d_head=128, R=8, K=8,
                         top_k=2, w=1024),
    "extreme_1m": Workload("extreme_1m", B=1, N=1048576, H=32, H_kv=8, d_head=128, R=1, K=4,
                           top_k=1, w=1024),
}


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 7919 + stream * 104729 + 17)
    return g


def _randn_bf16(shape, gen, device, chunk_elems: int = 1 << 28) -> torch.Tensor:
    """iid N(0,1) drawn in fp32 and rounded to bf16 (round-to-nearest-even), in chunks
    so that very large tensors never need a full fp32 temporary."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        flat[s:e] = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


def make_routing(wl: Workload, seed: int = 0, device="cpu"):
    """Routing vectors r [B, N, R, 16] fp32 and centroids C [K, 16] fp32."""
    if wl.routing == "proj768":
        gx = _gen(seed, 4, device)
        gw = _gen(seed, 5, device)
        x = torch.randn(wl.B * wl.N * wl.R, 768, generator=gx, device=device, dtype=torch.float64)
        W = torch.randn(768, D_G, generator=gw, device=device, dtype=torch.float64) / math.sqrt(768.0)
        r = (x @ W).to(torch.float32).view(wl.B, wl.N, wl.R, D_G)
    else:
        r = torch.randn(wl.B, wl.N, wl.R, D_G, generator=_gen(seed, 3, device), device=device,
                        dtype=torch.float32)
    C = torch.randn(wl.K, D_G, generator=_gen(seed, 6, device), device=device, dtype=torch.float32)
    return r.contiguous(), C.contiguous()


def make_qkv(wl: Workload, seed: int = 0, device="cpu"):
    """q [B, N, H, d], k and v [B, N, H_kv, d], bf16, iid N(0,1)."""
    q = _randn_bf16((wl.B, wl.N, wl.H, wl.d_head), _gen(seed, 0, device), device)
    k = _randn_bf16((wl.B, wl.N, wl.H_kv, wl.d_head), _gen(seed, 1, device), device)
    v = _randn_bf16((wl.B, wl.N, wl.H_kv, wl.d_head), _gen(seed, 2, device), device)
    return q, k, v


def make_inputs(wl: Workload, seed: int = 0, device="cpu") -> dict:
    q, k, v = make_qkv(wl, seed, device)
    r, C = make_routing(wl, seed, device)
    return {"q": q, "k": k, "v": v, "r": r, "C": C}


def sample_queries(N: int, n: int, w: int, seed: int = 0) -> torch.Tensor:
    """Seeded sample of n query positions in [0, N): always includes 0, w-1, w and N-1
    (where they exist), plus uniform draws without replacement; sorted, int64."""
    fixed = sorted({p for p in (0, w - 1, w, N - 1) if 0 <= p < N})
    if n >= N:
        return torch.arange(N, dtype=torch.int64)
    g = torch.Generator().manual_seed(seed * 31 + 7)
    picked = set(fixed)
    while len(picked) < n:
        cand = torch.randint(0, N, (2 * n,), generator=g).tolist()
        for c in cand:
            if len(picked) >= n:
                break
            picked.add(int(c))
    return torch.tensor(sorted(picked), dtype=torch.int64)
