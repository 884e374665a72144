"""Sharding one Focus attention problem over several GPUs with no exchange (host side).

Attention never mixes heads: query head h reads only KV head h / (H / H_kv) and
routing head (h / (H / H_kv)) / (H_kv / R), and the group masks of a routing head
depend only on its own routing vectors ("Why Attend to Everything? Focus is the
Key", gist.science technical summary, section 2 "Core Architecture": centroid
routing per token, attention inside the window and the shared groups).  So a
problem splits into independent sub-problems along the batch and along runs of
consecutive KV heads that hold whole routing heads; each rank computes its part
with the ordinary single-GPU entry points and nothing is exchanged.  With R = 1
the single routing head is needed by every rank and each recomputes it (routing
is a 64-byte read per token).
"""
from __future__ import annotations

import dataclasses


@dataclasses.dataclass(frozen=True)
class Shard:
    """One rank's part: batch rows [b0, b1), KV heads [kv0, kv1), query heads
    [h0, h1), routing heads [rho0, rho1); `empty` when the rank has no work."""
    b0: int
    b1: int
    kv0: int
    kv1: int
    h0: int
    h1: int
    rho0: int
    rho1: int

    @property
    def empty(self) -> bool:
        return self.b1 <= self.b0 or self.kv1 <= self.kv0


def _split(n: int, parts: int, i: int) -> tuple[int, int]:
    """Contiguous near-equal split of range(n) into `parts`; part i."""
    lo = n * i // parts
    hi = n * (i + 1) // parts
    return lo, hi


def shard(B: int, H: int, H_kv: int, R: int, world: int, rank: int) -> Shard:
    """The part of rank `rank` of `world`: the ranks are laid out as a grid of
    batch groups x head groups, with as many head groups as there are units of
    whole routing heads to go round (unit = H_kv / R KV heads when R > 1, one KV
    head when R = 1), and the batch split over the rest.  Ranks beyond the grid
    get an empty part."""
    if not (B >= 1 and H % H_kv == 0 and H_kv % R == 0 and 0 <= rank < world):
        raise ValueError("invalid shape or rank")
    unit = 1 if R == 1 else H_kv // R
    units = H_kv // unit
    n_head = min(units, world)
    while world % n_head:            # a grid that uses every rank where possible
        n_head -= 1
    n_batch = min(B, world // n_head)
    if rank >= n_head * n_batch:
        return Shard(0, 0, 0, 0, 0, 0, 0, 0)
    bi, hi = divmod(rank, n_head)
    b0, b1 = _split(B, n_batch, bi)
    u0, u1 = _split(units, n_head, hi)
    kv0, kv1 = u0 * unit, u1 * unit
    gq = H // H_kv
    if R == 1:
        rho0, rho1 = 0, 1
    else:
        rho0, rho1 = kv0 // unit, kv1 // unit
    return Shard(b0, b1, kv0, kv1, kv0 * gq, kv1 * gq, rho0, rho1)


def sub_params(p, s: Shard):
    """The single-GPU problem of shard s (a Params of the binding, or anything
    with the same fields and a dataclasses.replace-compatible type)."""
    return dataclasses.replace(p, B=s.b1 - s.b0, H=s.h1 - s.h0, H_kv=s.kv1 - s.kv0,
                               R=s.rho1 - s.rho0)


def slice_inputs(x: dict, s: Shard) -> dict:
    """The shard's inputs out of the full problem's tensors: q [B, N, H, d], k and v
    [B, N, H_kv, d], r [B, N, R, 16], C [K, 16] (shared)."""
    return {"q": x["q"][s.b0:s.b1, :, s.h0:s.h1].contiguous(),
            "k": x["k"][s.b0:s.b1, :, s.kv0:s.kv1].contiguous(),
            "v": x["v"][s.b0:s.b1, :, s.kv0:s.kv1].contiguous(),
            "r": x["r"][s.b0:s.b1, :, s.rho0:s.rho1].contiguous(),
            "C": x["C"]}
