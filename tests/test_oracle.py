"""Pins for the CPU oracle: each check ties it to something other than itself
(brute force, library routines, closed forms, invariants, printed values)."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _routing(B, N, R, K, seed):
    g = torch.Generator().manual_seed(seed)
    r = torch.randn(B, N, R, 16, generator=g, dtype=torch.float32)
    C = torch.randn(K, 16, generator=g, dtype=torch.float32)
    return r.numpy(), C.numpy()


def _bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


def _f64(t):
    return t.to(torch.float64).numpy()


# ------------------------------------------------------------------ routing ---

@pytest.mark.parametrize("K,top_k", [(4, 1), (4, 2), (5, 3), (8, 2), (6, 6)])
def test_scores_match_matmul_and_topk_is_best_subset(K, top_k):
    r, C = _routing(2, 96, 2, K, seed=K * 10 + top_k)
    mask, margin, kappa, beta = oracle.route(r, C, K=K, top_k=top_k)
    # scores: library matmul in fp64 on the same fp32 inputs
    s = np.einsum("bnrt,gt->brng", r.astype(np.float64), C.astype(np.float64))
    np.testing.assert_allclose(kappa, s, rtol=0, atol=1e-12)
    assert np.all(beta == 0.0)
    # membership: the k-subset with the largest total key (brute force over subsets)
    subsets = list(itertools.combinations(range(K), top_k))
    for b, rho, i in itertools.product(range(2), range(2), range(96)):
        best = max(subsets, key=lambda S: sum(s[b, rho, i, g] for g in S))
        assert mask[b, rho, i] == sum(1 << g for g in best)
        assert bin(int(mask[b, rho, i])).count("1") == top_k
        srt = np.sort(s[b, rho, i])[::-1]
        want = srt[top_k - 1] - srt[top_k] if top_k < K else math.inf
        assert margin[b, rho, i] == pytest.approx(want, abs=1e-12)


def test_topk_matches_stable_argsort_and_ties_go_low():
    r, C = _routing(1, 200, 1, 6, seed=3)
    C[4] = C[1]  # exact tie between groups 1 and 4 for every token
    mask, margin, kappa, _ = oracle.route(r, C, K=6, top_k=2)
    order = np.argsort(-kappa, axis=-1, kind="stable")[..., :2]
    want = np.bitwise_or.reduce((1 << order).astype(np.uint32), axis=-1)
    np.testing.assert_array_equal(mask, want)
    # where exactly one of the tied pair makes the cut, the lower index wins
    both = (mask >> 1) & 1, (mask >> 4) & 1
    assert np.all(both[1] <= both[0])
    assert np.any(both[0] != both[1])


def test_score_fp32_mode_is_fma_chain_and_close_to_fp64():
    r, C = _routing(1, 128, 1, 4, seed=5)
    _, _, k64, _ = oracle.route(r, C, K=4, top_k=2)
    _, _, k32, _ = oracle.route(r, C, K=4, top_k=2, score_fp32=True)
    # every fp32 key is an fp32 number within a few ulps of the exact dot product
    assert np.all(k32.astype(np.float32).astype(np.float64) == k32)
    np.testing.assert_allclose(k32, k64, rtol=0, atol=1e-5)
    # fused multiply-add chain, t = 0..15, emulated exactly: each fp32 fma is the
    # fp32 rounding of the exact product-sum (exact in fp64 for fp32 operands)
    i, g = 17, 2
    acc = np.float32(0)
    for t in range(16):
        acc = np.float32(np.float64(r[0, i, 0, t]) * np.float64(C[g, t]) + np.float64(acc))
    assert k32[0, 0, i, g] == float(acc)


def test_permuting_centroids_permutes_mask_bits():
    r, C = _routing(1, 300, 2, 5, seed=9)
    perm = np.array([3, 0, 4, 1, 2])
    m0, _, _, _ = oracle.route(r, C, K=5, top_k=2, sinkhorn_iters=2)
    m1, _, _, _ = oracle.route(r, C[perm], K=5, top_k=2, sinkhorn_iters=2)
    remap = np.zeros(m1.shape, np.int64)
    for new_g, old_g in enumerate(perm):
        remap |= ((m1.astype(np.int64) >> new_g) & 1) << int(old_g)
    np.testing.assert_array_equal(remap, m0)


def test_sinkhorn_zero_iterations_is_plain_topk():
    r, C = _routing(1, 256, 1, 4, seed=11)
    a, _, ka, _ = oracle.route(r, C, K=4, top_k=2, sinkhorn_iters=0, sinkhorn_eps=0.5)
    b, _, kb, _ = oracle.route(r, C, K=4, top_k=2)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(ka, kb)


def _implied_assignment(kappa):
    # row step applied to the oracle's keys: P_ig = exp(kappa_ig) / sum_g exp(kappa_ig)
    k = kappa - kappa.max(axis=-1, keepdims=True)
    p = np.exp(k)
    return p / p.sum(axis=-1, keepdims=True)


def test_sinkhorn_marginals_converge_to_balanced_groups():
    N, K = 600, 4
    r, C = _routing(1, N, 1, K, seed=13)
    C[0] *= 3.0  # strongly unbalanced raw scores
    devs = []
    for T in (1, 3, 10, 200):
        _, _, kappa, _ = oracle.route(r, C, K=K, top_k=1, sinkhorn_iters=T)
        P = _implied_assignment(kappa[0, 0])
        np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-12)
        devs.append(np.abs(P.sum(axis=0) - N / K).max())
    assert devs[0] > devs[1] > devs[2] > devs[3]
    assert devs[3] < 1e-6 * N


def test_sinkhorn_matches_probability_domain_matrix_scaling():
    """Sinkhorn-Knopp written as alternate column / row rescaling of exp(s/eps)."""
    N, K, T, eps = 40, 5, 4, 0.7
    r, C = _routing(1, N, 1, K, seed=17)
    mask, _, kappa, beta = oracle.route(r, C, K=K, top_k=2, sinkhorn_iters=T, sinkhorn_eps=eps)
    s = r[0, :, 0].astype(np.float64) @ C.astype(np.float64).T
    P = np.exp(s / eps)
    for _ in range(T):
        P = P * ((N / K) / P.sum(axis=0, keepdims=True))
        P = P / P.sum(axis=1, keepdims=True)
    logP = np.log(P)
    # same within-row ordering: log P - kappa is constant along each row
    d = logP - kappa[0, 0]
    np.testing.assert_allclose(d - d[:, :1], 0.0, atol=1e-10)
    order = np.argsort(-P, axis=1, kind="stable")[:, :2]
    want = np.bitwise_or.reduce((1 << order).astype(np.uint32), axis=1)
    np.testing.assert_array_equal(mask[0, 0], want)


def test_sinkhorn_first_column_potentials_closed_form():
    """One iteration: the row potentials are still zero at the column step, so
    beta_g = log(N / K) - log sum_i exp(s_ig / eps) exactly (target mass N / K per
    group; a constant shift of every beta_g would leave the masks unchanged, so only
    this pins the level)."""
    N, K, eps = 300, 5, 0.8
    r, C = _routing(2, N, 1, K, seed=29)
    _, _, _, beta = oracle.route(r, C, K=K, top_k=2, sinkhorn_iters=1, sinkhorn_eps=eps)
    s = np.einsum("bnt,gt->bng", r[:, :, 0].astype(np.float64), C.astype(np.float64)) / eps
    m = s.max(axis=1, keepdims=True)
    lse = (m + np.log(np.exp(s - m).sum(axis=1, keepdims=True)))[:, 0]
    np.testing.assert_allclose(beta[:, 0], math.log(N / K) - lse, atol=1e-12, rtol=0)


def test_sinkhorn_eps_is_a_score_scale():
    r, C = _routing(1, 300, 1, 4, seed=19)
    a, _, ka, _ = oracle.route(r, C, K=4, top_k=2, sinkhorn_iters=3, sinkhorn_eps=1.0)
    b, _, kb, _ = oracle.route(2.0 * r, C, K=4, top_k=2, sinkhorn_iters=3, sinkhorn_eps=2.0)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_allclose(ka, kb, atol=1e-9)


# ------------------------------------------------------------------- pairs ---

def _dense_allowed(mask_row, w):
    """N x N boolean matrix built from the definition, one pair at a time."""
    N = len(mask_row)
    A = np.zeros((N, N), bool)
    for i in range(N):
        for j in range(i + 1):
            A[i, j] = (i - j < w) or (int(mask_row[i]) & int(mask_row[j])) != 0
    return A


def test_allowed_pairs_brute_force_and_closed_forms():
    N, w = 130, 7
    rng = np.random.default_rng(0)
    mask = rng.integers(0, 16, size=(2, 3, N)).astype(np.uint32)
    cnt = oracle.allowed_pairs(mask, w)
    for b in range(2):
        for rho in range(3):
            assert cnt[b, rho] == _dense_allowed(mask[b, rho], w).sum()
    ones = np.ones((1, 1, N), np.uint32)
    assert oracle.allowed_pairs(ones, w)[0, 0] == N * (N + 1) // 2
    zeros = np.zeros((1, 1, N), np.uint32)
    assert oracle.allowed_pairs(zeros, w)[0, 0] == N * w - w * (w - 1) // 2


def test_table7_pairs_retained():
    """Printed 'pairs retained' for K=4: top-3 and top-4 keep every pair (any two
    3-subsets of 4 groups intersect); top-1 keeps sum_g p_g^2 = 1/4 of the distant
    pairs when Sinkhorn balances the groups (printed: 26% and 25%)."""
    gold = json.load(open(os.path.join(GOLDEN, "table7_pairs_retained.json")))
    N, K, w = 2048, gold["K"], 1
    r, C = _routing(1, N, 1, K, seed=23)
    causal = N * (N + 1) // 2
    for row in gold["rows"]:
        if row["top_k"] in (3, 4):
            m, _, _, _ = oracle.route(r, C, K=K, top_k=row["top_k"])
            assert oracle.allowed_pairs(m, w)[0, 0] / causal == row["pairs_retained"] == 1.0
    m, _, _, _ = oracle.route(r, C, K=K, top_k=1, sinkhorn_iters=30)
    frac = oracle.allowed_pairs(m, w)[0, 0] / causal
    printed = [row["pairs_retained"] for row in gold["rows"] if row["top_k"] == 1]
    assert min(printed) - 0.015 <= frac <= max(printed) + 0.015


# --------------------------------------------------------------- attention ---

def _dense_reference(q, k, v, mask, w, scale):
    """Dense masked softmax from an explicit N x N mask (fp64 numpy)."""
    B, N, H, d = q.shape
    H_kv = k.shape[2]
    R = mask.shape[1]
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    o = np.zeros((B, N, H, d))
    lse = np.zeros((B, N, H))
    for b in range(B):
        for h in range(H):
            kvh = h // (H // H_kv)
            rho = kvh // (H_kv // R)
            A = _dense_allowed(mask[b, rho], w)
            S = scale * qf[b, :, h] @ kf[b, :, kvh].T
            S = np.where(A, S, -np.inf)
            m = S.max(axis=1, keepdims=True)
            e = np.exp(S - m)
            l = e.sum(axis=1, keepdims=True)
            o[b, :, h] = (e / l) @ vf[b, :, kvh]
            lse[b, :, h] = (m + np.log(l))[:, 0]
    return o.reshape(B * N, H, d), lse.reshape(B * N, H)


@pytest.mark.parametrize("B,N,H,H_kv,R,d,K,top_k,w", [
    (1, 70, 2, 2, 1, 16, 4, 2, 5),
    (2, 97, 4, 2, 2, 8, 5, 1, 9),
    (1, 64, 4, 1, 1, 32, 3, 1, 1),
    (1, 50, 2, 2, 2, 8, 8, 3, 64),
    (1, 60, 8, 4, 2, 8, 4, 2, 5),  # two KV heads per routing head: the routing-head map shows
])
def test_attention_matches_dense_masked_softmax(B, N, H, H_kv, R, d, K, top_k, w):
    q, k, v = _bf16((B, N, H, d), 1), _bf16((B, N, H_kv, d), 2), _bf16((B, N, H_kv, d), 3)
    r, C = _routing(B, N, R, K, seed=4)
    mask, _, _, _ = oracle.route(r, C, K=K, top_k=top_k)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attn(q, k, v, mask, w=w)
    o_ref, lse_ref = _dense_reference(q, k, v, mask, w, scale)
    np.testing.assert_allclose(o, o_ref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-12, rtol=0)


def _sdpa_causal(q, k, v):
    """torch's dense causal attention in fp64, [B, N, H, d] in and out."""
    H, H_kv = q.shape[2], k.shape[2]
    qt = q.to(torch.float64).transpose(1, 2)
    kt = k.to(torch.float64).repeat_interleave(H // H_kv, dim=2).transpose(1, 2)
    vt = v.to(torch.float64).repeat_interleave(H // H_kv, dim=2).transpose(1, 2)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
    return o.transpose(1, 2).reshape(-1, H, q.shape[3]).numpy()


@pytest.mark.parametrize("case", ["K1", "topk_eq_K", "pigeonhole", "window_covers"])
def test_special_cases_reduce_to_dense_causal(case):
    B, N, H, H_kv, d = 1, 150, 4, 2, 32
    K, top_k, w = {"K1": (1, 1, 3), "topk_eq_K": (4, 4, 2), "pigeonhole": (5, 3, 4),
                   "window_covers": (4, 1, 150)}[case]
    q, k, v = _bf16((B, N, H, d), 5), _bf16((B, N, H_kv, d), 6), _bf16((B, N, H_kv, d), 7)
    r, C = _routing(B, N, 1, K, seed=8)
    mask, _, _, _ = oracle.route(r, C, K=K, top_k=top_k)
    o, lse = oracle.attn(q, k, v, mask, w=w)
    np.testing.assert_allclose(o, _sdpa_causal(q, k, v), atol=1e-12, rtol=0)
    assert oracle.allowed_pairs(mask, w)[0, 0] == N * (N + 1) // 2


def test_unit_window_top1_is_per_group_causal_attention():
    """w=1, top_k=1: each query sees itself and earlier tokens of its own group only,
    i.e. dense causal attention on each group's gathered subsequence."""
    B, N, H, d, K = 1, 180, 2, 16, 4
    q, k, v = _bf16((B, N, H, d), 9), _bf16((B, N, H, d), 10), _bf16((B, N, H, d), 11)
    r, C = _routing(B, N, 1, K, seed=12)
    mask, _, _, _ = oracle.route(r, C, K=K, top_k=1)
    o, _ = oracle.attn(q, k, v, mask, w=1)
    for g in range(K):
        idx = np.nonzero(mask[0, 0] == (1 << g))[0]
        if len(idx) == 0:
            continue
        sel = torch.from_numpy(idx)
        ref = _sdpa_causal(q[:, sel], k[:, sel], v[:, sel])
        np.testing.assert_allclose(o[idx], ref, atol=1e-12, rtol=0)


def test_identical_keys_reveal_the_attended_set():
    """All keys equal, v_j = e_j: O_i = 1/|A_i| on exactly the union set A_i, and
    LSE_i = scale q_i.k + log |A_i|. Hand-checkable sets on a small case."""
    N, w = 24, 3
    # groups of each token (K=3, up to two groups each)
    mask = np.array([[[1, 2, 4, 1, 3, 2, 4, 5, 1, 6, 2, 4, 1, 1, 2, 3, 4, 6, 5, 1, 2, 4, 7, 1]]],
                    np.uint32)
    d = N
    q = _bf16((1, N, 1, d), 13)
    krow = _bf16((1, 1, 1, d), 14)
    k = krow.expand(1, N, 1, d).contiguous()
    v = torch.eye(N, dtype=torch.bfloat16).view(1, N, 1, d)
    o, lse = oracle.attn(q, k, v, mask, w=w, scale=0.25)
    m = mask[0, 0].tolist()
    for i in range(N):
        A = {j for j in range(i + 1) if i - j < w or (m[i] & m[j])}
        want = np.array([1.0 / len(A) if j in A else 0.0 for j in range(N)])
        np.testing.assert_allclose(o[i, 0], want, atol=1e-15)
        s = 0.25 * float((q[0, i, 0].double() * krow[0, 0, 0].double()).sum())
        assert lse[i, 0] == pytest.approx(s + math.log(len(A)), abs=1e-12)


def test_rows_sum_to_one_and_union_lse_dominates_window():
    B, N, H, d = 1, 200, 2, 16
    q, k = _bf16((B, N, H, d), 15), _bf16((B, N, H, d), 16)
    ones = torch.ones(B, N, H, d, dtype=torch.bfloat16)
    r, C = _routing(B, N, 1, 4, seed=17)
    mask, _, _, _ = oracle.route(r, C, K=4, top_k=2)
    o, lse = oracle.attn(q, k, ones, mask, w=8)
    np.testing.assert_allclose(o, 1.0, atol=1e-13)
    _, lse_win = oracle.attn(q, k, ones, np.zeros_like(mask), w=8)
    assert np.all(lse >= lse_win - 1e-13)
    assert np.any(lse > lse_win + 1e-3)


def test_row_subset_equals_full_rows():
    wl = synth.WORKLOADS["tiny"].replace(N=160)
    x = synth.make_inputs(wl, seed=1)
    mask, _, _, _ = oracle.route(x["r"], x["C"], K=wl.K, top_k=wl.top_k)
    o, lse = oracle.attn(x["q"], x["k"], x["v"], mask, w=wl.w)
    rows = synth.sample_queries(wl.N, 20, wl.w, seed=2)
    os_, ls_ = oracle.attn(x["q"], x["k"], x["v"], mask, w=wl.w, rows=rows)
    np.testing.assert_array_equal(os_, o[rows.numpy()])
    np.testing.assert_array_equal(ls_, lse[rows.numpy()])


# ---------------------------------------------------------------- backward ---

def _loss(q, k, v, mask, G, w):
    """L = sum O * G with the forward oracle (fp64)."""
    o, _ = oracle.attn(q, k, v, mask, w=w)
    return float((o * G).sum())


def _bf16_neighbours(x: torch.Tensor):
    """The two bf16 values adjacent to the bf16 scalar x (below, above)."""
    bits = x.view(torch.int16).item()
    a = torch.tensor([bits - 1], dtype=torch.int16).view(torch.bfloat16)[0]
    b = torch.tensor([bits + 1], dtype=torch.int16).view(torch.bfloat16)[0]
    return (a, b) if float(a) < float(b) else (b, a)


def test_gradients_match_central_differences_between_adjacent_bf16_values():
    """dL/dx ~ (L(x+) - L(x-)) / (x+ - x-) with x+- the bf16 neighbours of x: the
    inputs stay exact, and the step (about 2^-8 |x|) leaves a truncation error far
    below the tolerance.  General mask: window and shared groups, GQA."""
    B, N, H, H_kv, d, K, top_k, w = 1, 48, 2, 1, 8, 4, 2, 5
    q, k, v = _bf16((B, N, H, d), 21), _bf16((B, N, H_kv, d), 22), _bf16((B, N, H_kv, d), 23)
    dout = _bf16((B, N, H, d), 24)
    G = _f64(dout).reshape(B * N, H, d)
    r, C = _routing(B, N, 1, K, seed=25)
    mask, _, _, _ = oracle.route(r, C, K=K, top_k=top_k)
    dq, dk, dv = oracle.attn_bwd(q, k, v, mask, dout, w=w)
    dq, dk, dv = dq.reshape(B, N, H, d), dk.reshape(B, N, H_kv, d), dv.reshape(B, N, H_kv, d)
    rng = np.random.default_rng(26)
    checked = 0
    for name, t, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in t.shape)
            x = t[idx]
            if not 0.25 < abs(float(x)) < 4.0:
                continue
            lo, hi = _bf16_neighbours(x)
            tl, th = t.clone(), t.clone()
            tl[idx], th[idx] = lo, hi
            args_l = {"q": q, "k": k, "v": v} | {name: tl}
            args_h = {"q": q, "k": k, "v": v} | {name: th}
            fd = (_loss(args_h["q"], args_h["k"], args_h["v"], mask, G, w)
                  - _loss(args_l["q"], args_l["k"], args_l["v"], mask, G, w)) / (float(hi) - float(lo))
            assert fd == pytest.approx(grad[idx], rel=2e-3, abs=2e-5), (name, idx)
            checked += 1
    assert checked >= 8


def _sdpa_grads(q, k, v, dout):
    """torch autograd of dense causal attention (fp64), [B, N, H(_kv), d] layouts."""
    H, H_kv = q.shape[2], k.shape[2]
    qt = q.to(torch.float64).requires_grad_()
    kt = k.to(torch.float64).requires_grad_()
    vt = v.to(torch.float64).requires_grad_()
    rep = lambda x: x.repeat_interleave(H // H_kv, dim=2).transpose(1, 2)
    o = torch.nn.functional.scaled_dot_product_attention(qt.transpose(1, 2), rep(kt), rep(vt),
                                                         is_causal=True)
    (o.transpose(1, 2) * dout.to(torch.float64)).sum().backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


@pytest.mark.parametrize("case", ["K1", "topk_eq_K", "window_covers"])
def test_gradients_reduce_to_dense_causal_autograd(case):
    B, N, H, H_kv, d = 2, 90, 4, 2, 16
    K, top_k, w = {"K1": (1, 1, 3), "topk_eq_K": (3, 3, 2), "window_covers": (4, 1, 90)}[case]
    q, k, v = _bf16((B, N, H, d), 31), _bf16((B, N, H_kv, d), 32), _bf16((B, N, H_kv, d), 33)
    dout = _bf16((B, N, H, d), 34)
    r, C = _routing(B, N, 1, K, seed=35)
    mask, _, _, _ = oracle.route(r, C, K=K, top_k=top_k)
    dq, dk, dv = oracle.attn_bwd(q, k, v, mask, dout, w=w)
    gq, gk, gv = _sdpa_grads(q, k, v, dout)
    np.testing.assert_allclose(dq, gq.reshape(B * N, H, d), atol=1e-11, rtol=0)
    np.testing.assert_allclose(dk, gk.reshape(B * N, H_kv, d), atol=1e-11, rtol=0)
    np.testing.assert_allclose(dv, gv.reshape(B * N, H_kv, d), atol=1e-11, rtol=0)


def test_unit_window_top1_gradients_are_per_group_causal_autograd():
    B, N, H, d, K = 1, 120, 2, 16, 4
    q, k, v = _bf16((B, N, H, d), 41), _bf16((B, N, H, d), 42), _bf16((B, N, H, d), 43)
    dout = _bf16((B, N, H, d), 44)
    r, C = _routing(B, N, 1, K, seed=45)
    mask, _, _, _ = oracle.route(r, C, K=K, top_k=1)
    dq, dk, dv = oracle.attn_bwd(q, k, v, mask, dout, w=1)
    for g in range(K):
        idx = np.nonzero(mask[0, 0] == (1 << g))[0]
        if len(idx) == 0:
            continue
        sel = torch.from_numpy(idx)
        gq, gk, gv = _sdpa_grads(q[:, sel], k[:, sel], v[:, sel], dout[:, sel])
        np.testing.assert_allclose(dq[idx], gq[0], atol=1e-11, rtol=0)
        np.testing.assert_allclose(dk[idx], gk[0], atol=1e-11, rtol=0)
        np.testing.assert_allclose(dv[idx], gv[0], atol=1e-11, rtol=0)


def _dense_masked_grads(q, k, v, mask, dout, w, scale):
    """torch autograd (fp64) through an explicit masked softmax, one (b, h) at a time,
    with the attended set built from the definition for h's routing head."""
    B, N, H, d = q.shape
    H_kv, R = k.shape[2], mask.shape[1]
    qt = q.to(torch.float64).requires_grad_()
    kt = k.to(torch.float64).requires_grad_()
    vt = v.to(torch.float64).requires_grad_()
    g = dout.to(torch.float64)
    loss = torch.zeros((), dtype=torch.float64)
    for b in range(B):
        for h in range(H):
            kvh = h // (H // H_kv)
            rho = kvh // (H_kv // R)
            A = torch.from_numpy(_dense_allowed(mask[b, rho], w))
            S = (scale * qt[b, :, h] @ kt[b, :, kvh].T).masked_fill(~A, float("-inf"))
            loss = loss + ((torch.softmax(S, dim=1) @ vt[b, :, kvh]) * g[b, :, h]).sum()
    loss.backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


@pytest.mark.parametrize("B,N,H,H_kv,R,d,K,top_k,w", [
    (1, 60, 8, 4, 2, 8, 4, 2, 5), (2, 45, 4, 2, 1, 16, 5, 2, 3)])
def test_gradients_match_dense_masked_softmax_autograd(B, N, H, H_kv, R, d, K, top_k, w):
    """General masks, GQA and several routing heads: the oracle's gradients against
    torch autograd through the dense masked softmax."""
    q, k, v = _bf16((B, N, H, d), 91), _bf16((B, N, H_kv, d), 92), _bf16((B, N, H_kv, d), 93)
    dout = _bf16((B, N, H, d), 94)
    r, C = _routing(B, N, R, K, seed=95)
    mask, _, _, _ = oracle.route(r, C, K=K, top_k=top_k)
    dq, dk, dv = oracle.attn_bwd(q, k, v, mask, dout, w=w)
    gq, gk, gv = _dense_masked_grads(q, k, v, mask, dout, w, 1.0 / math.sqrt(d))
    np.testing.assert_allclose(dq, gq.reshape(B * N, H, d), atol=1e-11, rtol=0)
    np.testing.assert_allclose(dk, gk.reshape(B * N, H_kv, d), atol=1e-11, rtol=0)
    np.testing.assert_allclose(dv, gv.reshape(B * N, H_kv, d), atol=1e-11, rtol=0)


@pytest.mark.parametrize("B,N,H,H_kv,R,d,K,top_k,w", [
    (2, 80, 4, 2, 2, 8, 5, 2, 6), (1, 130, 3, 1, 1, 16, 8, 3, 17)])
def test_gradient_sum_rules(B, N, H, H_kv, R, d, K, top_k, w):
    """Softmax rows: sum_j dS_ij = 0, so the dk of a KV head sum to zero over its keys;
    sum_j P_ij = 1, so its dv sum to the dO of the queries that read it."""
    q, k, v = _bf16((B, N, H, d), 51), _bf16((B, N, H_kv, d), 52), _bf16((B, N, H_kv, d), 53)
    dout = _bf16((B, N, H, d), 54)
    r, C = _routing(B, N, R, K, seed=55)
    mask, _, _, _ = oracle.route(r, C, K=K, top_k=top_k)
    _, dk, dv = oracle.attn_bwd(q, k, v, mask, dout, w=w)
    dk, dv = dk.reshape(B, N, H_kv, d), dv.reshape(B, N, H_kv, d)
    g = _f64(dout).reshape(B, N, H_kv, H // H_kv, d).sum(axis=3)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=1), g.sum(axis=1), atol=1e-11)


def test_gradient_subsets_equal_full_computation():
    wl = synth.WORKLOADS["tiny"].replace(N=150, H=4, H_kv=2)
    x = synth.make_inputs(wl, seed=3)
    dout = _bf16((1, wl.N, wl.H, wl.d_head), 61)
    mask, _, _, _ = oracle.route(x["r"], x["C"], K=wl.K, top_k=wl.top_k)
    dq, dk, dv = oracle.attn_bwd(x["q"], x["k"], x["v"], mask, dout, w=wl.w)
    rows = synth.sample_queries(wl.N, 12, wl.w, seed=4)
    keys = synth.sample_queries(wl.N, 9, wl.w, seed=5)
    dq_s, dk_s, dv_s = oracle.attn_bwd(x["q"], x["k"], x["v"], mask, dout, w=wl.w, rows=rows,
                                       keys=keys, heads=[2, 3])
    np.testing.assert_allclose(dq_s, dq[rows.numpy()][:, [2, 3]], atol=1e-12, rtol=0)
    # KV head 1 is read by query heads 2 and 3 only
    np.testing.assert_allclose(dk_s[:, 1], dk[keys.numpy(), 1], atol=1e-12, rtol=0)
    np.testing.assert_allclose(dv_s[:, 1], dv[keys.numpy(), 1], atol=1e-12, rtol=0)
    assert np.all(dk_s[:, 0] == 0) and np.all(dv_s[:, 0] == 0)


def test_gradients_with_given_forward_output_shift_as_the_d_term_predicts():
    """dq_i = scale sum_j P_ij (dP_ij - D_i) k_j is affine in D_i: taking D'_i = dO_i . R_i
    from a given array R moves dq_i by -scale (D'_i - D_i) (P k)_i, where (P k)_i is the
    forward with v := k, and leaves dv unchanged.  R varies per row and head, so a
    wrong index into it shows."""
    B, N, H, H_kv, d, K, top_k, w = 2, 60, 4, 2, 16, 4, 2, 7
    q, k, v = _bf16((B, N, H, d), 71), _bf16((B, N, H_kv, d), 72), _bf16((B, N, H_kv, d), 73)
    dout = _bf16((B, N, H, d), 74)
    R = _bf16((B, N, H, d), 75)
    r, C = _routing(B, N, 1, K, seed=76)
    mask, _, _, _ = oracle.route(r, C, K=K, top_k=top_k)
    dq0, dk0, dv0 = oracle.attn_bwd(q, k, v, mask, dout, w=w)
    dq1, _, dv1 = oracle.attn_bwd(q, k, v, mask, dout, w=w, o_for_D=R)
    o, _ = oracle.attn(q, k, v, mask, w=w)
    pk, _ = oracle.attn(q, k, k, mask, w=w)
    g = _f64(dout).reshape(B * N, H, d)
    D = (g * o).sum(axis=2)
    D1 = (g * _f64(R).reshape(B * N, H, d)).sum(axis=2)
    scale = 1.0 / math.sqrt(d)
    np.testing.assert_allclose(dq1 - dq0, -scale * (D1 - D)[:, :, None] * pk, atol=1e-11, rtol=0)
    np.testing.assert_allclose(dv1, dv0, atol=1e-13, rtol=0)


def test_gradient_magnitudes_bound_the_gradients_and_reduce_without_d_term():
    """mq, mk, mv sum the absolute values of the terms of dq, dk, dv, so they bound
    them; with d_rel = 0 and a single allowed key per row (w = 1, one group per
    token in its own group) dS = 0 and mq = mk = 0, mv_j = |dO_j|."""
    B, N, H, H_kv, d, K, top_k, w = 1, 70, 2, 1, 16, 4, 2, 6
    q, k, v = _bf16((B, N, H, d), 81), _bf16((B, N, H_kv, d), 82), _bf16((B, N, H_kv, d), 83)
    dout = _bf16((B, N, H, d), 84)
    r, C = _routing(B, N, 1, K, seed=85)
    mask, _, _, _ = oracle.route(r, C, K=K, top_k=top_k)
    dq, dk, dv, mq, mk, mv = oracle.attn_bwd(q, k, v, mask, dout, w=w, magnitudes=True, d_rel=1.0)
    assert np.all(np.abs(dq) <= mq + 1e-12) and np.all(np.abs(dk) <= mk + 1e-12)
    assert np.all(np.abs(dv) <= mv + 1e-12)
    n = 30
    lone = (1 << np.arange(n)).astype(np.uint32)[None, None, :]   # every token its own group
    q, k, v, dout = q[:, :n].contiguous(), k[:, :n].contiguous(), v[:, :n].contiguous(), dout[:, :n].contiguous()
    dq, dk, dv, mq, mk, mv = oracle.attn_bwd(q, k, v, lone, dout, w=1, magnitudes=True)
    assert np.all(mq == 0) and np.all(mk == 0)
    np.testing.assert_allclose(mv[:, 0], np.abs(_f64(dout)[0]).sum(axis=1), atol=1e-14, rtol=0)
