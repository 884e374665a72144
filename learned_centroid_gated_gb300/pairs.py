"""Exact count of allowed (query, key) pairs, for FLOP accounting (host side).

A pair (i, j) is allowed when j <= i and either i - j < w (window) or the two
tokens' group bitmasks intersect ("Why Attend to Everything? Focus is the Key",
gist.science technical summary, section 2, "Inference Efficiency (Top-k)").
The count is exact: window pairs in closed form, long-range pairs by binary
search of each query position minus w in the sorted positions of every
compatible mask value.  O(N log N * distinct masks), no N x N work.
"""
from __future__ import annotations

import numpy as np


def window_pairs(N: int, w: int) -> int:
    """sum_i min(i + 1, w) for i < N."""
    if N <= w:
        return N * (N + 1) // 2
    return N * w - w * (w - 1) // 2


def allowed_pairs(mask, w: int) -> np.ndarray:
    """mask [B, R, N] (uint32 bit patterns, any integer dtype) -> [B, R] int64 counts."""
    m = np.asarray(mask).astype(np.int64) & 0xFFFFFFFF
    B, R, N = m.shape
    out = np.zeros((B, R), np.int64)
    win = window_pairs(N, w)
    for b in range(B):
        for rho in range(R):
            row = m[b, rho]
            vals, inv = np.unique(row, return_inverse=True)
            pos = [np.nonzero(inv == a)[0] for a in range(len(vals))]  # ascending
            far = 0
            for a, va in enumerate(vals):
                qpos = pos[a] - w  # keys j <= i - w
                for c, vc in enumerate(vals):
                    if int(va) & int(vc):
                        far += int(np.searchsorted(pos[c], qpos, side="right").sum())
            out[b, rho] = win + far
    return out


def allowed_flops(mask, w: int, H: int, H_kv: int, d_head: int) -> int:
    """4 * d_head FLOPs per allowed pair per query head (QK^T and PV, 2 each)."""
    cnt = allowed_pairs(mask, w)  # [B, R]
    R = cnt.shape[1]
    heads_per_rho = H // R
    return int(4 * d_head * heads_per_rho * cnt.sum())


def executed_tiles(mask, w: int, block_rows: int = 256, key_tile: int = 128,
                   group_lists: bool = False):
    """Key tiles the tensor-core kernels run, per (b, routing head), for FLOP
    accounting of executed (not just allowed) work: long-range = for every block of
    `block_rows` consecutive rows of one mask value, ceil(keys / key_tile) over each
    compatible mask value's keys with pos <= (last row's pos) - w (with group_lists:
    blocks of each group's list against that list's keys); window = for every block
    of `block_rows` consecutive tokens, ceil(span / key_tile) with span the keys
    (first row - w, last row], one fewer for a full block past the first w - 1 tokens
    with two or more key tiles (its two halves skip the band's last and first key tile
    respectively).  Counts are in block_rows x key_tile tiles.  Returns
    (long_tiles [B, R], window_tiles)."""
    m = np.asarray(mask).astype(np.int64) & 0xFFFFFFFF
    B, R, N = m.shape
    long_t = np.zeros((B, R), np.int64)
    for b in range(B):
        for rho in range(R):
            row = m[b, rho]
            if group_lists:
                for g in range(32):
                    pos = np.nonzero((row >> g) & 1)[0]
                    if len(pos) == 0:
                        continue
                    last = pos[np.minimum(np.arange(block_rows - 1, len(pos) + block_rows - 1,
                                                    block_rows), len(pos) - 1)]
                    cnt = np.searchsorted(pos, last - w, side="right")
                    long_t[b, rho] += int(((cnt + key_tile - 1) // key_tile).sum())
                continue
            vals, inv = np.unique(row, return_inverse=True)
            pos = [np.nonzero(inv == a)[0] for a in range(len(vals))]
            for a, va in enumerate(vals):
                last = pos[a][np.minimum(np.arange(block_rows - 1, len(pos[a]) + block_rows - 1,
                                                   block_rows), len(pos[a]) - 1)]
                for c, vc in enumerate(vals):
                    if int(va) & int(vc):
                        cnt = np.searchsorted(pos[c], last - w, side="right")
                        long_t[b, rho] += int(((cnt + key_tile - 1) // key_tile).sum())
    starts = np.arange(0, N, block_rows)
    ends = np.minimum(starts + block_rows, N)
    span = ends - np.maximum(0, starts - w + 1)
    n_win = (span + key_tile - 1) // key_tile
    skew = (starts >= w - 1) & (ends - starts == block_rows) & (n_win >= 2)
    win_t = int((n_win - skew).sum())
    return long_t, win_t
