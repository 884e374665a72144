"""Focus centroid-gated sparse attention for GB300 (sm_103a): routing, the forward
pass (exact-set segments or group lists), decode, and the backward pass with the
group masks held fixed.

Thin ctypes binding over the C ABI in ``include/focus.h`` (``libfocus.so``, built
in-tree by ``learned_centroid_gated_gb300.build``). This module only marshals
arguments: every step of the computation runs in the library's CUDA kernels.
PyTorch supplies device memory and streams. There is no CPU fallback: importing
this package fails if the library is missing.

Method: "Why Attend to Everything? Focus is the Key" -- gist.science technical
summary, section 2 "Core Architecture" and "Inference Efficiency (Top-k)".
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# FOCUS_DEBUG_BOUNDS=1: the debug build (index checks raise FOCUS_ERR_BOUNDS; build it
# with the same variable set), else the default build
LIB_PATH = os.path.join(_HERE, "libfocus_debug.so" if os.environ.get("FOCUS_DEBUG_BOUNDS", "")
                        not in ("", "0") else "libfocus.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "focus.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"Focus CUDA library not built ({LIB_PATH} missing); run "
        "`python learned_centroid_gated_gb300/build.py` on a machine with nvcc")

_lib = ctypes.CDLL(LIB_PATH)

FOCUS_OK = 0
ERRORS = {
    -1: "FOCUS_ERR_INVALID_ARG", -2: "FOCUS_ERR_UNSUPPORTED", -3: "FOCUS_ERR_WORKSPACE",
    -4: "FOCUS_ERR_CUDA", -5: "FOCUS_ERR_TIMEOUT", -6: "FOCUS_ERR_BOUNDS", -7: "FOCUS_ERR_ALIGNMENT",
    -8: "FOCUS_ERR_NONFINITE",
}


class FocusError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        detail = strerror(code)
        if code == -4:  # FOCUS_ERR_CUDA: name the CUDA error behind it
            detail += ": " + _lib.focus_cuda_error_string().decode()
        super().__init__(f"{what}: {ERRORS.get(code, code)} ({detail})")


class _Params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("B", "N", "H", "H_kv", "d_head", "R", "K", "top_k", "w", "sinkhorn_iters")] + \
               [("sinkhorn_eps", ctypes.c_float), ("softmax_scale", ctypes.c_float),
                ("schedule", ctypes.c_int32)]

SCHEDULE_AUTO, SCHEDULE_SEGMENTS, SCHEDULE_GROUPS = 0, 1, 2


@dataclasses.dataclass(frozen=True)
class Params:
    """Problem description (focus_params).  softmax_scale <= 0 selects 1/sqrt(d_head);
    schedule: SCHEDULE_AUTO, SCHEDULE_SEGMENTS (exact group sets) or SCHEDULE_GROUPS
    (one list per group)."""
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
    softmax_scale: float = 0.0
    schedule: int = 0

    @classmethod
    def from_workload(cls, wl, **kw) -> "Params":
        return cls(B=wl.B, N=wl.N, H=wl.H, H_kv=wl.H_kv, d_head=wl.d_head, R=wl.R, K=wl.K,
                   top_k=wl.top_k, w=wl.w, sinkhorn_iters=wl.sinkhorn_iters,
                   sinkhorn_eps=wl.sinkhorn_eps, **kw)

    def c(self) -> _Params:
        return _Params(*[getattr(self, f.name) for f in dataclasses.fields(self)])

    @property
    def nseg(self) -> int:
        """Segments of the bucketing that runs: C(K, top_k) exact sets, or K lists."""
        return self.bucket_shape()[1]

    def bucket_shape(self):
        """(schedule that runs, segments, permuted rows per (b, routing head))."""
        nseg, rows = ctypes.c_int32(), ctypes.c_int32()
        rc = _lib.focus_bucket_shape(ctypes.byref(self.c()), ctypes.byref(nseg), ctypes.byref(rows))
        _check(rc if rc < 0 else 0, "focus_bucket_shape")
        return rc, nseg.value, rows.value

    @property
    def scale(self) -> float:
        return self.softmax_scale if self.softmax_scale > 0 else 1.0 / math.sqrt(self.d_head)


_P = ctypes.c_void_p
_PP = ctypes.POINTER(_Params)
_lib.focus_workspace_size.argtypes = [_PP]
_lib.focus_workspace_size.restype = ctypes.c_size_t
_lib.focus_route.argtypes = [_PP, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
_lib.focus_route.restype = ctypes.c_int
_lib.focus_bucket_shape.argtypes = [_PP, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
_lib.focus_bucket_shape.restype = ctypes.c_int
_lib.focus_bucket.argtypes = [_PP, _P, _P, _P, _P, ctypes.c_size_t, _P]
_lib.focus_bucket.restype = ctypes.c_int
_lib.focus_attn_fwd.argtypes = [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
_lib.focus_attn_fwd.restype = ctypes.c_int
_lib.focus_attn_fwd_ev.argtypes = [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P,
                                   ctypes.POINTER(ctypes.c_void_p)]
_lib.focus_attn_fwd_ev.restype = ctypes.c_int
N_STAGE_EVENTS = 6
STAGES = ("route", "bucket", "permute", "attn_window", "attn_long")
_lib.focus_route_static.argtypes = [_PP, _P, _P, _P, _P, _P]
_lib.focus_route_static.restype = ctypes.c_int
_lib.focus_route_static_limit.argtypes = []
_lib.focus_route_static_limit.restype = ctypes.c_size_t
_lib.focus_bwd_workspace_size.argtypes = [_PP]
_lib.focus_bwd_workspace_size.restype = ctypes.c_size_t
_lib.focus_attn_bwd.argtypes = [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
_lib.focus_attn_bwd.restype = ctypes.c_int
_lib.focus_attn_bwd_ev.argtypes = [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P,
                                   ctypes.POINTER(ctypes.c_void_p)]
_lib.focus_attn_bwd_ev.restype = ctypes.c_int
N_BWD_STAGE_EVENTS = 5
BWD_STAGES = ("prepare", "window", "long_dq", "long_dkdv")
_lib.focus_decode_workspace_size.argtypes = [_PP]
_lib.focus_decode_workspace_size.restype = ctypes.c_size_t
_lib.focus_decode.argtypes = [_PP, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
_lib.focus_decode.restype = ctypes.c_int
_lib.focus_selftest_timeout.argtypes = [_P, ctypes.c_size_t, _P]
_lib.focus_selftest_timeout.restype = ctypes.c_int
_lib.focus_get_status.argtypes = [_P, _P]
_lib.focus_get_status.restype = ctypes.c_int
_lib.focus_strerror.argtypes = [ctypes.c_int]
_lib.focus_strerror.restype = ctypes.c_char_p
_lib.focus_version.argtypes = []
_lib.focus_version.restype = ctypes.c_int
_lib.focus_cuda_error_string.argtypes = []
_lib.focus_cuda_error_string.restype = ctypes.c_char_p


def declared_symbols() -> list[str]:
    """Function names declared in include/focus.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(focus_\w+)\s*\(", text, re.M)))


def strerror(code: int) -> str:
    return _lib.focus_strerror(code).decode()


def version() -> int:
    return _lib.focus_version()


def workspace_size(p: Params) -> int:
    return int(_lib.focus_workspace_size(ctypes.byref(p.c())))


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int, what: str):
    if rc != FOCUS_OK:
        raise FocusError(rc, what)


class Workspace:
    """Caller-owned device workspace (a torch uint8 buffer), grown on demand."""

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.buf: torch.Tensor | None = None

    def get(self, p: Params) -> torch.Tensor:
        need = workspace_size(p)
        if need == 0:
            raise FocusError(-1, "focus_workspace_size")
        if self.buf is None or self.buf.numel() < need:
            self.buf = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self.buf


_default_ws: dict = {}


def _ws(p: Params, ws, device) -> torch.Tensor:
    if isinstance(ws, torch.Tensor):
        return ws
    if ws is None:
        ws = _default_ws.setdefault(str(device), Workspace(device))
    return ws.get(p)


def _bf16_bits(t: torch.Tensor) -> torch.Tensor:
    assert t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous()
    return t


def route(p: Params, r: torch.Tensor, C: torch.Tensor, *, margin: bool = False, ws=None,
          stream=None):
    """Group bitmasks [B, R, N] uint32 (as int32 tensor) and optional fp32 margins."""
    assert r.dtype == torch.float32 and C.dtype == torch.float32 and r.is_cuda and C.is_cuda
    mask = torch.empty(p.B, p.R, p.N, dtype=torch.int32, device=r.device)
    marg = torch.empty(p.B, p.R, p.N, dtype=torch.float32, device=r.device) if margin else None
    w = _ws(p, ws, r.device)
    _check(_lib.focus_route(ctypes.byref(p.c()), _ptr(r.contiguous()), _ptr(C.contiguous()),
                            _ptr(mask), _ptr(marg), _ptr(w), w.numel(), _stream(stream)),
           "focus_route")
    return mask, marg


def route_static_limit() -> int:
    """Bytes of the fixed device scratch that route_static uses for Sinkhorn."""
    return int(_lib.focus_route_static_limit())


def route_static(p: Params, r: torch.Tensor, C: torch.Tensor, *, margin: bool = False,
                 stream=None):
    """route() without a workspace: the library's fixed device scratch
    (route_static_limit() bytes, used by the Sinkhorn step only) is used instead,
    for callers that must not allocate device memory when they call in.  The
    outputs here are still torch tensors; pass preallocated ones through the C ABI
    (focus_route_static) to allocate nothing at all."""
    assert r.dtype == torch.float32 and C.dtype == torch.float32 and r.is_cuda and C.is_cuda
    mask = torch.empty(p.B, p.R, p.N, dtype=torch.int32, device=r.device)
    marg = torch.empty(p.B, p.R, p.N, dtype=torch.float32, device=r.device) if margin else None
    _check(_lib.focus_route_static(ctypes.byref(p.c()), _ptr(r.contiguous()), _ptr(C.contiguous()),
                                   _ptr(mask), _ptr(marg), _stream(stream)), "focus_route_static")
    return mask, marg


def bucket(p: Params, mask: torch.Tensor, *, ws=None, stream=None):
    """Stable bucketing: perm [B, R, rows] int32 and seg_off [B, R, nseg+1] int32, where
    (nseg, rows) = (C(K, top_k), N) for exact-set segments and (K, N * top_k) for group lists."""
    _, nseg, rows = p.bucket_shape()
    perm = torch.empty(p.B, p.R, rows, dtype=torch.int32, device=mask.device)
    seg = torch.empty(p.B, p.R, nseg + 1, dtype=torch.int32, device=mask.device)
    w = _ws(p, ws, mask.device)
    _check(_lib.focus_bucket(ctypes.byref(p.c()), _ptr(mask.contiguous()), _ptr(perm), _ptr(seg),
                             _ptr(w), w.numel(), _stream(stream)), "focus_bucket")
    return perm, seg


def attn_fwd(p: Params, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, r=None, C=None,
             mask=None, *, out=None, lse=None, want_lse: bool = True, ws=None, stream=None,
             stage_events=None):
    """Focus attention forward on device tensors. Returns (o bf16 [B,N,H,d], lse fp32 [B,H,N]).

    stage_events: optional list of N_STAGE_EVENTS torch.cuda.Event(enable_timing=True),
    recorded at the stage boundaries (see focus_attn_fwd_ev)."""
    for t in (q, k, v):
        _bf16_bits(t)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(p.B, p.H, p.N, dtype=torch.float32, device=q.device)
    w = _ws(p, ws, q.device)
    args = (ctypes.byref(p.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(r), _ptr(C), _ptr(mask), _ptr(out),
            _ptr(lse), _ptr(w), w.numel(), _stream(stream))
    if stage_events is None:
        _check(_lib.focus_attn_fwd(*args), "focus_attn_fwd")
    else:
        assert len(stage_events) == N_STAGE_EVENTS
        for e in stage_events:
            if e.cuda_event == 0:  # torch creates the CUDA event on its first record
                e.record(stream or torch.cuda.current_stream())
        evs = (ctypes.c_void_p * N_STAGE_EVENTS)(*[e.cuda_event for e in stage_events])
        _check(_lib.focus_attn_fwd_ev(*args, evs), "focus_attn_fwd_ev")
    return out, lse


_lib.focus_host_workspace_size.argtypes = [_PP, ctypes.c_int]
_lib.focus_host_workspace_size.restype = ctypes.c_size_t
_lib.focus_attn_fwd_host.argtypes = [_PP, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int, _P, ctypes.c_size_t,
                                     _P, _P]
_lib.focus_attn_fwd_host.restype = ctypes.c_int
_lib.focus_host_groups.argtypes = [_PP, ctypes.c_int, ctypes.POINTER(ctypes.c_int32), ctypes.c_int]
_lib.focus_host_groups.restype = ctypes.c_int


def host_groups(p: Params, n_groups: int = 0) -> list[int]:
    """KV heads of each head group focus_attn_fwd_host uses (in order)."""
    buf = (ctypes.c_int32 * 64)()
    n = _lib.focus_host_groups(ctypes.byref(p.c()), n_groups, buf, 64)
    _check(n if n < 0 else 0, "focus_host_groups")
    return list(buf[:n])


def host_workspace_size(p: Params, n_groups: int = 0) -> int:
    return int(_lib.focus_host_workspace_size(ctypes.byref(p.c()), n_groups))


class HostSession:
    """End-to-end calls on HOST tensors through focus_attn_fwd_host: the heads are
    processed in groups, copies of one group overlapping the compute of another, on
    two streams of this session.  Inputs should be pinned (tensor.pin_memory()) for
    the copies to overlap.  Each call returns pinned host tensors (o, lse) that the
    next call overwrites."""

    def __init__(self, p: Params, device="cuda", n_groups: int = 0):
        self.p = p
        self.device = torch.device(device)
        self.n_groups = n_groups
        need = host_workspace_size(p, n_groups)
        if need == 0:
            raise FocusError(-1, "focus_host_workspace_size")
        self.ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        self.compute = torch.cuda.Stream(self.device)
        self.copy = torch.cuda.Stream(self.device)
        self.o_host = torch.empty(p.B, p.N, p.H, p.d_head, dtype=torch.bfloat16, pin_memory=True)
        self.lse_host = torch.empty(p.B, p.H, p.N, dtype=torch.float32, pin_memory=True)

    def group_sizes(self) -> list[int]:
        """KV heads of each head group, in processing order."""
        return host_groups(self.p, self.n_groups)

    def h2d_bytes(self, *tensors) -> int:
        return sum(t.numel() * t.element_size() for t in tensors)

    def d2h_bytes(self) -> int:
        return self.o_host.numel() * 2 + self.lse_host.numel() * 4

    def __call__(self, q, k, v, r, C):
        for t, dt in ((q, torch.bfloat16), (k, torch.bfloat16), (v, torch.bfloat16),
                      (r, torch.float32), (C, torch.float32)):
            assert t.device.type == "cpu" and t.dtype == dt and t.is_contiguous()
        _check(_lib.focus_attn_fwd_host(ctypes.byref(self.p.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(r),
                                        _ptr(C), _ptr(self.o_host), _ptr(self.lse_host), self.n_groups,
                                        _ptr(self.ws), self.ws.numel(),
                                        ctypes.c_void_p(self.compute.cuda_stream),
                                        ctypes.c_void_p(self.copy.cuda_stream)),
               "focus_attn_fwd_host")
        self.copy.synchronize()
        return self.o_host, self.lse_host


def attn_fwd_host(p: Params, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, r: torch.Tensor,
                  C: torch.Tensor, *, device="cuda", n_groups: int = 0):
    """One end-to-end call on HOST tensors (see HostSession for repeated calls).
    Returns host (o, lse)."""
    o, lse = HostSession(p, device, n_groups)(q, k, v, r, C)
    return o.clone(), lse.clone()


def decode_workspace_size(p: Params) -> int:
    return int(_lib.focus_decode_workspace_size(ctypes.byref(p.c())))


def decode(p: Params, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
           mask: torch.Tensor, *, out=None, lse=None, want_lse: bool = True, ws=None, stream=None):
    """Decode step for the newest token of each sequence (position p.N - 1).
    q [B, H, d] bf16; caches [B, N, H_kv, d] bf16 (newest token included); mask
    [B, R, N] (int32 view of uint32).  Returns (o [B, H, d] bf16, lse [B, H] fp32)."""
    for t in (q, k_cache, v_cache):
        _bf16_bits(t)
    if out is None:
        out = torch.empty(p.B, p.H, p.d_head, dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty(p.B, p.H, dtype=torch.float32, device=q.device)
    need = decode_workspace_size(p)
    if need == 0:
        raise FocusError(-1, "focus_decode_workspace_size")
    if ws is None or ws.numel() < need:
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(_lib.focus_decode(ctypes.byref(p.c()), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                             _ptr(mask.contiguous()), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                             _stream(stream)), "focus_decode")
    return out, lse


def bwd_workspace_size(p: Params) -> int:
    return int(_lib.focus_bwd_workspace_size(ctypes.byref(p.c())))


def attn_bwd(p: Params, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: torch.Tensor,
             o: torch.Tensor, lse: torch.Tensor, d_o: torch.Tensor, *, dq=None, dk=None, dv=None,
             ws=None, stream=None, stage_events=None):
    """Backward of attn_fwd with the masks held fixed.  q, o, d_o [B, N, H, d] bf16;
    k, v [B, N, H_kv, d] bf16; mask [B, R, N] (the forward's); lse [B, H, N] fp32 (the
    forward's).  Returns (dq, dk, dv) bf16 in the layouts of q, k, v.

    stage_events: optional list of N_BWD_STAGE_EVENTS torch.cuda.Event(enable_timing=True)
    recorded at the stage boundaries (see focus_attn_bwd_ev)."""
    for t in (q, k, v, o, d_o):
        _bf16_bits(t)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = bwd_workspace_size(p)
    if need == 0:
        raise FocusError(-2, "focus_bwd_workspace_size")
    if ws is None or ws.numel() < need:
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    args = (ctypes.byref(p.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(mask.contiguous()), _ptr(o),
            _ptr(lse.contiguous()), _ptr(d_o), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(),
            _stream(stream))
    if stage_events is None:
        _check(_lib.focus_attn_bwd(*args), "focus_attn_bwd")
    else:
        assert len(stage_events) == N_BWD_STAGE_EVENTS
        for e in stage_events:
            if e.cuda_event == 0:  # torch creates the CUDA event on its first record
                e.record(stream or torch.cuda.current_stream())
        evs = (ctypes.c_void_p * N_BWD_STAGE_EVENTS)(*[e.cuda_event for e in stage_events])
        _check(_lib.focus_attn_bwd_ev(*args, evs), "focus_attn_bwd_ev")
    return dq, dk, dv


def selftest_timeout(device="cuda", stream=None) -> int:
    """Run the device failure-path diagnostic; returns the status (-5 = FOCUS_ERR_TIMEOUT)."""
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=device)
    return _lib.focus_selftest_timeout(_ptr(ws), ws.numel(), _stream(stream))


def get_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronise and read the device status word of the last call on `ws`."""
    return _lib.focus_get_status(_ptr(ws), _stream(stream))
