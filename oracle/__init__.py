"""CPU fp64 oracle for Focus centroid-gated sparse attention (forward and backward).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline leg, never by the CUDA library or its Python binding.
The arithmetic lives in ``focus_oracle.c`` (plain C, fp64); this module compiles it
with gcc into ``liboracle.so`` next to the source and marshals numpy arrays.

Parity pins (tests/test_oracle.py): top-k against brute force over all k-subsets
and against numpy's stable sort; Sinkhorn against its marginal constraints and a
probability-domain restatement; the attended set against a dense N x N mask built
from the definition; values against dense causal attention in the cases that
reduce to it (K=1, top_k=K, 2*top_k>K, w>=N) and against per-group causal
attention for w=1, top_k=1; rows of the softmax sum to one.  Gradients: central
differences of the forward between adjacent bf16 values, torch autograd of dense
causal attention in the cases that reduce to it, per-group causal attention for
w=1, top_k=1, and the sum rules sum_j dk_j = 0, sum_j dv_j = sum_i dO_i.  The Sinkhorn step's
agreement with the authors' own (unpublished) formula is parity unpinned: the
pages give no formula and no numbers for it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "focus_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, so results match across hosts)."""
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                                   "-pthread", _SRC, "-o", tmp, "-lm"])
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _open(path: str):
    """The oracle library at `path` with its entry points' signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, f64, i64 = ctypes.c_int, ctypes.c_double, ctypes.c_int64
    lib.oracle_route.argtypes = [i32, i32, i32, i32, i32, i32, f64, i32, P, P, P, P, P, P]
    lib.oracle_route.restype = i32
    lib.oracle_allowed_pairs.argtypes = [i32, i32, i32, i32, P, P]
    lib.oracle_allowed_pairs.restype = i32
    lib.oracle_attn.argtypes = [i32, i32, i32, i32, i32, i32, i32, f64, P, P, P, P, P, i64, P, i32,
                                P, P, i32]
    lib.oracle_attn.restype = i32
    lib.oracle_attn_bwd.argtypes = [i32, i32, i32, i32, i32, i32, i32, f64, P, P, P, P, P, P, P,
                                    i64, P, i64, P, i32, P, P, P, P, P, P, f64, i32]
    lib.oracle_attn_bwd.restype = i32
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _open(_LIB_PATH)
    return _lib


def compile_variant(source: str, out_path: str) -> str:
    """Compile a variant of the oracle's C source with the same flags (tests plant
    mistakes in copies of the source to check that the pins reject them)."""
    src_path = out_path[:-3] + ".c" if out_path.endswith(".so") else out_path + ".c"
    with open(src_path, "w") as f:
        f.write(source)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                           "-pthread", src_path, "-o", out_path, "-lm"])
    return out_path


class use_library:
    """Context manager: the module's functions call the library at `path` inside it."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = _load()
        _lib = _open(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def n_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _np(x, dtype) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().cpu()
        if str(x.dtype) == "torch.bfloat16":
            x = x.view(__import__("torch").int16).numpy().view(np.uint16)
        else:
            x = x.numpy()
    return np.ascontiguousarray(x, dtype=dtype)


def route(r, C, *, K: int, top_k: int, sinkhorn_iters: int = 0, sinkhorn_eps: float = 1.0,
          score_fp32: bool = False):
    """Scores, optional Sinkhorn and top-k for r [B, N, R, 16] and C [K, 16].

    Returns (mask [B, R, N] uint32, margin [B, R, N] f64, kappa [B, R, N, K] f64,
    beta [B, R, K] f64)."""
    r = _np(r, np.float32)
    C = _np(C, np.float32)
    B, N, R, dg = r.shape
    assert dg == 16 and C.shape == (K, 16)
    mask = np.zeros((B, R, N), np.uint32)
    margin = np.zeros((B, R, N), np.float64)
    kappa = np.zeros((B, R, N, K), np.float64)
    beta = np.zeros((B, R, K), np.float64)
    rc = _load().oracle_route(B, N, R, K, top_k, sinkhorn_iters, sinkhorn_eps, int(score_fp32),
                              _ptr(r), _ptr(C), _ptr(mask), _ptr(margin), _ptr(kappa), _ptr(beta))
    if rc != 0:
        raise ValueError("oracle_route: bad arguments")
    return mask, margin, kappa, beta


def allowed_pairs(mask, w: int) -> np.ndarray:
    """Brute-force count of allowed (i, j) pairs per (b, routing head): [B, R] int64."""
    mask = _np(mask, np.uint32)
    B, R, N = mask.shape
    out = np.zeros((B, R), np.int64)
    if _load().oracle_allowed_pairs(B, N, R, w, _ptr(mask), _ptr(out)) != 0:
        raise ValueError("oracle_allowed_pairs: bad arguments")
    return out


def attn(q, k, v, mask, *, w: int, scale: float | None = None, rows=None, heads=None,
         n_threads: int | None = None):
    """Union-softmax attention for q [B, N, H, d], k/v [B, N, H_kv, d] (bf16 tensors or
    uint16 bit arrays) and mask [B, R, N].

    rows: optional flattened query rows (b * N + i); heads: optional query heads.
    Returns (o [n_rows, n_heads, d] f64, lse [n_rows, n_heads] f64)."""
    q16, k16, v16 = _np(q, np.uint16), _np(k, np.uint16), _np(v, np.uint16)
    mask = _np(mask, np.uint32)
    B, N, H, d = q16.shape
    H_kv = k16.shape[2]
    R = mask.shape[1]
    assert k16.shape == (B, N, H_kv, d) and v16.shape == k16.shape and mask.shape == (B, R, N)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows_a = None if rows is None else _np(rows, np.int64)
    n_rows = B * N if rows_a is None else rows_a.shape[0]
    heads_a = None if heads is None else _np(heads, np.int32)
    n_heads = H if heads_a is None else heads_a.shape[0]
    o = np.zeros((n_rows, n_heads, d), np.float64)
    lse = np.zeros((n_rows, n_heads), np.float64)
    rc = _load().oracle_attn(B, N, H, H_kv, R, d, w, float(scale), _ptr(q16), _ptr(k16), _ptr(v16),
                             _ptr(mask), _ptr(rows_a), n_rows, _ptr(heads_a), n_heads, _ptr(o),
                             _ptr(lse), n_threads or n_cores())
    if rc != 0:
        raise ValueError("oracle_attn: bad arguments")
    return o, lse


def attn_bwd(q, k, v, mask, dout, *, w: int, scale: float | None = None, rows=None, keys=None,
             heads=None, o_for_D=None, magnitudes: bool = False, d_rel: float = 0.0,
             n_threads: int | None = None):
    """Gradients of ``attn`` with the mask held fixed, for upstream gradient dout
    [B, N, H, d] (bf16 tensor or uint16 bits).

    rows: flattened query rows (b * N + i) whose dq is wanted (default all);
    keys: flattened key rows (b * N + j) whose dk, dv are wanted (default all);
    heads: query heads differentiated (default all); dk, dv sum over them.
    o_for_D: optional bf16 forward output [B, N, H, d]; D_i = dO_i . o_i is then taken
    from it (as an implementation that receives o in bf16 does) instead of the exact
    sum_j P_ij dP_ij.
    magnitudes: also return (mq, mk, mv), first-order error scales: the sums of the
    absolute values of the gradient's terms, where each dS_ij (and P_ij for dv) is
    widened by d_rel times the absolute sums that form its logit, dP_ij and D_i (see
    oracle_attn_bwd in focus_oracle.c); a relative error u in those steps moves a
    gradient by about u times its scale.
    Returns (dq [n_rows, n_heads, d], dk [n_keys, H_kv, d], dv [n_keys, H_kv, d]), f64."""
    q16, k16, v16, g16 = (_np(t, np.uint16) for t in (q, k, v, dout))
    o16 = None if o_for_D is None else _np(o_for_D, np.uint16)
    mask = _np(mask, np.uint32)
    B, N, H, d = q16.shape
    H_kv = k16.shape[2]
    R = mask.shape[1]
    assert g16.shape == q16.shape and k16.shape == (B, N, H_kv, d) and v16.shape == k16.shape
    assert o16 is None or o16.shape == q16.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows_a = None if rows is None else _np(rows, np.int64)
    keys_a = None if keys is None else _np(keys, np.int64)
    heads_a = None if heads is None else _np(heads, np.int32)
    n_rows = B * N if rows_a is None else rows_a.shape[0]
    n_keys = B * N if keys_a is None else keys_a.shape[0]
    n_heads = H if heads_a is None else heads_a.shape[0]
    dq = np.zeros((n_rows, n_heads, d), np.float64)
    dk = np.zeros((n_keys, H_kv, d), np.float64)
    dv = np.zeros((n_keys, H_kv, d), np.float64)
    mq = np.zeros_like(dq) if magnitudes else None
    mk = np.zeros_like(dk) if magnitudes else None
    mv = np.zeros_like(dv) if magnitudes else None
    rc = _load().oracle_attn_bwd(B, N, H, H_kv, R, d, w, float(scale), _ptr(q16), _ptr(k16), _ptr(v16),
                                 _ptr(mask), _ptr(g16), _ptr(o16), _ptr(rows_a), n_rows, _ptr(keys_a), n_keys,
                                 _ptr(heads_a), n_heads, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(mq),
                                 _ptr(mk), _ptr(mv), float(d_rel), n_threads or n_cores())
    if rc != 0:
        raise ValueError("oracle_attn_bwd: bad arguments")
    if magnitudes:
        return dq, dk, dv, mq, mk, mv
    return dq, dk, dv
