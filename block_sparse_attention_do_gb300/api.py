"""ctypes binding over libnsa.so (declared in include/nsa.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  torch provides device memory (outputs and the
workspace) and the current CUDA stream.  There is no CPU fallback: if the
library is missing the first call raises.
"""
from __future__ import annotations

import ctypes as C
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnsa.so")

NSA_OK = 0
STATUS = {0: "NSA_OK", 1: "NSA_ERR_INVALID_ARG", 2: "NSA_ERR_UNSUPPORTED", 3: "NSA_ERR_BAD_INDEX",
          4: "NSA_ERR_DEVICE_TIMEOUT", 5: "NSA_ERR_CUDA", 6: "NSA_ERR_WORKSPACE"}
DTYPE = {torch.float32: 0, torch.bfloat16: 1}
LAYOUT_BHTD, LAYOUT_THD = 0, 1

# every entry point of include/nsa.h
SYMBOLS = (
    "nsa_fwd_workspace_size", "nsa_bwd_workspace_size", "nsa_sel_fwd", "nsa_sel_bwd",
    "nsa_dense_causal_fwd", "nsa_dense_causal_bwd", "nsa_sel_varlen_fwd", "nsa_sel_varlen_bwd",
    "nsa_do_dot", "nsa_inverse_index_offsets_len", "nsa_build_inverse_index", "nsa_get_error",
    "nsa_status_string", "nsa_count_pairs", "nsa_trace_enable", "nsa_trace_reset",
    "nsa_trace_count", "nsa_trace_get", "nsa_build_inverse_index_noalloc",
    "nsa_plan_size", "nsa_plan_build", "nsa_bwd_planned_workspace_size", "nsa_sel_bwd_planned",
    "nsa_swa_fwd", "nsa_swa_bwd", "nsa_sink_fwd", "nsa_sink_bwd", "nsa_debug_stall",
    "nsa_causal_fwd_workspace_size", "nsa_causal_bwd_workspace_size", "nsa_causal_fwd", "nsa_causal_bwd",
    "nsa_select_workspace_size", "nsa_compress_keys_mean", "nsa_block_scores", "nsa_select_topk",
    "nsa_sel_fwd_workspace_size", "nsa_sel_bwd_workspace_size",
)


class Problem(C.Structure):
    _fields_ = [("B", C.c_int32), ("Hq", C.c_int32), ("Hkv", C.c_int32), ("T", C.c_int32),
                ("D", C.c_int32), ("block_size", C.c_int32), ("S", C.c_int32),
                ("dtype", C.c_int32), ("layout", C.c_int32), ("total_tokens", C.c_int32),
                ("scale", C.c_float), ("reserved", C.c_int32),
                ("q_stride", C.c_int64 * 3), ("kv_stride", C.c_int64 * 3), ("o_stride", C.c_int64 * 3),
                ("dq_stride", C.c_int64 * 3), ("dkv_stride", C.c_int64 * 3),
                ("Tk", C.c_int32), ("total_keys", C.c_int32), ("bottom_right", C.c_int32),
                ("reserved2", C.c_int32)]


def _bht_strides(t, thd):
    """(batch, head, token) element strides of a [B, H, T, D] (or packed
    [total, H, D]) tensor whose last dimension is contiguous."""
    if t.stride(-1) != 1:
        raise ValueError("the head dimension must be contiguous")
    if thd:
        return (0, t.stride(1), t.stride(0))
    return (t.stride(0), t.stride(1), t.stride(2))


def declare_strides(p: Problem, thd: bool, q=None, k=None, o=None, dq=None, dk=None) -> Problem:
    """Fills the problem's declared strides from the tensors given (k stands
    for k and v, o for o and dO, dk for dk and dv)."""
    for name, t in (("q_stride", q), ("kv_stride", k), ("o_stride", o), ("dq_stride", dq),
                    ("dkv_stride", dk)):
        if t is not None:
            getattr(p, name)[:] = _bht_strides(t, thd)
    return p


def _same_strides(a, b, what):
    if a is not None and b is not None and a.stride() != b.stride():
        raise ValueError(f"{what} must have the same strides")


class NsaError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


_lib = None
_P = C.c_void_p


def lib() -> C.CDLL:
    """Load libnsa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libnsa.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = C.CDLL(LIB_PATH)
        pp = C.POINTER(Problem)
        L.nsa_fwd_workspace_size.restype = C.c_size_t
        L.nsa_fwd_workspace_size.argtypes = [pp]
        L.nsa_bwd_workspace_size.restype = C.c_size_t
        L.nsa_bwd_workspace_size.argtypes = [pp]
        L.nsa_sel_fwd.argtypes = [pp] + [_P] * 6 + [_P, C.c_size_t, _P]
        L.nsa_sel_bwd.argtypes = [pp] + [_P] * 10 + [_P, C.c_size_t, _P]
        L.nsa_dense_causal_fwd.argtypes = [pp] + [_P] * 5 + [_P, C.c_size_t, _P]
        L.nsa_dense_causal_bwd.argtypes = [pp] + [_P] * 9 + [_P, C.c_size_t, _P]
        L.nsa_sel_varlen_fwd.argtypes = [pp] + [_P] * 7 + [_P, C.c_size_t, _P]
        L.nsa_sel_varlen_bwd.argtypes = [pp] + [_P] * 11 + [_P, C.c_size_t, _P]
        L.nsa_do_dot.argtypes = [pp] + [_P] * 4 + [_P]
        L.nsa_inverse_index_offsets_len.restype = C.c_int64
        L.nsa_inverse_index_offsets_len.argtypes = [pp]
        L.nsa_build_inverse_index.argtypes = [pp] + [_P] * 4 + [_P, C.c_size_t, _P]
        L.nsa_get_error.argtypes = [_P, _P, C.POINTER(C.c_int32)]
        L.nsa_status_string.restype = C.c_char_p
        L.nsa_status_string.argtypes = [C.c_int32]
        L.nsa_count_pairs.argtypes = [pp] + [_P] * 3 + [_P]
        L.nsa_build_inverse_index_noalloc.argtypes = [pp] + [_P] * 5 + [_P]
        L.nsa_plan_size.restype = C.c_size_t
        L.nsa_plan_size.argtypes = [pp]
        L.nsa_plan_build.argtypes = [pp, _P, _P, _P, C.c_size_t, _P]
        L.nsa_bwd_planned_workspace_size.restype = C.c_size_t
        L.nsa_bwd_planned_workspace_size.argtypes = [pp]
        L.nsa_sel_bwd_planned.argtypes = [pp] + [_P] * 12 + [_P, C.c_size_t, _P]
        L.nsa_swa_fwd.argtypes = [pp, C.c_int32] + [_P] * 6 + [_P, C.c_size_t, _P]
        L.nsa_swa_bwd.argtypes = [pp, C.c_int32] + [_P] * 10 + [_P, C.c_size_t, _P]
        L.nsa_sink_fwd.argtypes = [pp, C.c_int32] + [_P] * 7 + [_P, C.c_size_t, _P]
        L.nsa_sink_bwd.argtypes = [pp, C.c_int32] + [_P] * 12 + [_P, C.c_size_t, _P]
        L.nsa_debug_stall.argtypes = [C.c_int32, C.c_int32]
        L.nsa_causal_fwd_workspace_size.restype = C.c_size_t
        L.nsa_causal_fwd_workspace_size.argtypes = [pp]
        L.nsa_causal_bwd_workspace_size.restype = C.c_size_t
        L.nsa_causal_bwd_workspace_size.argtypes = [pp]
        L.nsa_causal_fwd.argtypes = [pp, C.c_int32] + [_P] * 7 + [_P, C.c_size_t, _P]
        L.nsa_causal_bwd.argtypes = [pp, C.c_int32] + [_P] * 11 + [_P, C.c_size_t, _P]
        L.nsa_trace_enable.argtypes = [C.c_int32]
        L.nsa_trace_reset.restype = None
        L.nsa_trace_reset.argtypes = []
        L.nsa_trace_count.restype = C.c_int32
        L.nsa_trace_count.argtypes = []
        L.nsa_trace_get.argtypes = [C.c_int32, C.POINTER(C.c_char_p), C.POINTER(C.c_float)]
        for name in ("nsa_sel_fwd_workspace_size", "nsa_sel_bwd_workspace_size"):
            getattr(L, name).restype = C.c_size_t
            getattr(L, name).argtypes = [pp]
        L.nsa_select_workspace_size.restype = C.c_size_t
        L.nsa_select_workspace_size.argtypes = [pp]
        L.nsa_compress_keys_mean.argtypes = [pp] + [_P] * 3 + [_P]
        L.nsa_block_scores.argtypes = [pp] + [_P] * 4 + [_P, C.c_size_t, _P]
        L.nsa_select_topk.argtypes = [pp] + [_P] * 3 + [_P]
        for name in SYMBOLS:
            fn = getattr(L, name)
            if fn.restype is C.c_int:  # default restype: status enums
                fn.restype = C.c_int32
        _lib = L
    return _lib


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _check(status, where):
    if status != NSA_OK:
        raise NsaError(status, where)


def problem(B, Hq, Hkv, T, D, block_size, S, dtype, layout=LAYOUT_BHTD, total_tokens=0,
            scale=None) -> Problem:
    return Problem(B, Hq, Hkv, T, D, block_size, S, DTYPE[dtype], layout, total_tokens,
                   float(scale) if scale else 0.0)


def problem_from(q, k, block_size, S, scale=None, cu_seqlens=None, max_seqlen=None) -> Problem:
    if cu_seqlens is None:
        B, Hq, T, D = q.shape
        return problem(B, Hq, k.shape[1], T, D, block_size, S, q.dtype, scale=scale)
    total, Hq, D = q.shape
    B = cu_seqlens.numel() - 1
    if max_seqlen is None:
        max_seqlen = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()) if B > 0 else 1
    return problem(B, Hq, k.shape[1], max(1, max_seqlen), D, block_size, S, q.dtype,
                   layout=LAYOUT_THD, total_tokens=total, scale=scale)


_ws_cache: dict = {}


def workspace(nbytes: int, device, key="default") -> torch.Tensor:
    """A cached device buffer of at least nbytes (256-byte aligned by torch)."""
    ck = (key, str(device))
    buf = _ws_cache.get(ck)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[ck] = buf
    return buf


def fwd_workspace_size(p: Problem) -> int:
    return int(lib().nsa_fwd_workspace_size(C.byref(p)))


def bwd_workspace_size(p: Problem) -> int:
    return int(lib().nsa_bwd_workspace_size(C.byref(p)))


def bwd_planned_workspace_size(p: Problem) -> int:
    return int(lib().nsa_bwd_planned_workspace_size(C.byref(p)))


def _lse_shape(q, cu_seqlens):
    return q.shape[:-1]


def sel_fwd(q, k, v, block_idx, block_size, scale=None, cu_seqlens=None, max_seqlen=None,
            dense=False, ws=None, stream=None, window=None, sinks=None):
    """Selection (or dense causal, or with `window` sliding-window causal)
    forward through the C ABI: returns (o, lse).  `sinks` (fp32, one logit
    per query head, dense entry only) adds attention sinks."""
    dense = dense or window is not None or sinks is not None
    S = 1 if dense else block_idx.shape[-1]
    p = problem_from(q, k, block_size, S, scale, cu_seqlens, max_seqlen)
    o = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    _same_strides(k, v, "k and v")
    declare_strides(p, cu_seqlens is not None, q=q, k=k, o=o)
    lse = torch.empty(_lse_shape(q, cu_seqlens), dtype=torch.float32, device=q.device)
    n = fwd_workspace_size(p)
    if n == 0:
        raise NsaError(1, "nsa_fwd_workspace_size")
    ws = workspace(n, q.device, "fwd") if ws is None else ws
    L = lib()
    st = _stream(stream)
    if sinks is not None:
        s = L.nsa_sink_fwd(C.byref(p), int(window or 0), _ptr(cu_seqlens), _ptr(sinks), _ptr(q), _ptr(k),
                           _ptr(v), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), st)
    elif window is not None:
        s = L.nsa_swa_fwd(C.byref(p), int(window), _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                          _ptr(lse), _ptr(ws), ws.numel(), st)
    elif cu_seqlens is not None:
        s = L.nsa_sel_varlen_fwd(C.byref(p), _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v),
                                 _ptr(block_idx), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), st)
    elif dense:
        s = L.nsa_dense_causal_fwd(C.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                   _ptr(ws), ws.numel(), st)
    else:
        s = L.nsa_sel_fwd(C.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(block_idx), _ptr(o),
                          _ptr(lse), _ptr(ws), ws.numel(), st)
    _check(s, "nsa fwd")
    return o, lse


def build_plan(q, k, block_idx, block_size, scale=None, cu_seqlens=None, max_seqlen=None,
               stream=None):
    """A reusable backward plan (device uint8 tensor) of block_idx, for
    sel_bwd(..., plan=...); q and k only give the problem's shapes."""
    p = problem_from(q, k, block_size, block_idx.shape[-1], scale, cu_seqlens, max_seqlen)
    L = lib()
    n = int(L.nsa_plan_size(C.byref(p)))
    if n == 0:
        raise NsaError(1, "nsa_plan_size")
    plan = torch.empty(n, dtype=torch.uint8, device=block_idx.device)
    _check(L.nsa_plan_build(C.byref(p), _ptr(cu_seqlens), _ptr(block_idx), _ptr(plan), plan.numel(),
                            _stream(stream)), "nsa_plan_build")
    return plan


def sel_bwd(q, k, v, o, dO, lse, block_idx, block_size, scale=None, cu_seqlens=None,
            max_seqlen=None, dense=False, ws=None, stream=None, out=None, plan=None, window=None,
            sinks=None):
    """Selection (or dense causal, or with `window` sliding-window causal)
    backward through the C ABI: returns (dq, dk, dv), and dsinks as a fourth
    value with `sinks` (dense entry only; o and lse as the sink forward wrote
    them).  With `plan` (from build_plan on the same block_idx) the index
    build is skipped."""
    dense = dense or window is not None or sinks is not None
    S = 1 if dense else block_idx.shape[-1]
    p = problem_from(q, k, block_size, S, scale, cu_seqlens, max_seqlen)
    if out is None:
        dq = torch.empty(q.shape, dtype=q.dtype, device=q.device)
        dk = torch.empty(k.shape, dtype=k.dtype, device=k.device)
        dv = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    else:
        dq, dk, dv = out
    _same_strides(k, v, "k and v")
    _same_strides(o, dO, "o and dO")
    _same_strides(dk, dv, "dk and dv")
    declare_strides(p, cu_seqlens is not None, q=q, k=k, o=o, dq=dq, dk=dk)
    L = lib()
    if plan is not None:
        if dense:
            raise ValueError("a plan serves the selection backward only")
        n = bwd_planned_workspace_size(p)
        if n == 0:
            raise NsaError(1, "nsa_bwd_planned_workspace_size")
        ws = workspace(n, q.device, "bwd_planned") if ws is None else ws
        s = L.nsa_sel_bwd_planned(C.byref(p), _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                  _ptr(dO), _ptr(lse), _ptr(block_idx), _ptr(plan), _ptr(dq), _ptr(dk),
                                  _ptr(dv), _ptr(ws), ws.numel(), _stream(stream))
        _check(s, "nsa_sel_bwd_planned")
        return dq, dk, dv
    n = bwd_workspace_size(p)
    if n == 0:
        raise NsaError(1, "nsa_bwd_workspace_size")
    ws = workspace(n, q.device, "bwd") if ws is None else ws
    st = _stream(stream)
    if sinks is not None:
        dsinks = torch.empty_like(sinks)
        s = L.nsa_sink_bwd(C.byref(p), int(window or 0), _ptr(cu_seqlens), _ptr(sinks), _ptr(q), _ptr(k),
                           _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dsinks),
                           _ptr(ws), ws.numel(), st)
        _check(s, "nsa_sink_bwd")
        return dq, dk, dv, dsinks
    if window is not None:
        s = L.nsa_swa_bwd(C.byref(p), int(window), _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                          _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(), st)
    elif cu_seqlens is not None:
        s = L.nsa_sel_varlen_bwd(C.byref(p), _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                 _ptr(dO), _ptr(lse), _ptr(block_idx), _ptr(dq), _ptr(dk),
                                 _ptr(dv), _ptr(ws), ws.numel(), st)
    elif dense:
        s = L.nsa_dense_causal_bwd(C.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO),
                                   _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(),
                                   st)
    else:
        s = L.nsa_sel_bwd(C.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse),
                          _ptr(block_idx), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(), st)
    _check(s, "nsa bwd")
    return dq, dk, dv


def _causal_problem(q, k, cu_q, cu_k, max_q, max_k, bottom_right, scale):
    if cu_q is None:
        B, Hq, T, D = q.shape
        p = problem(B, Hq, k.shape[1], T, D, 64, 1, q.dtype, scale=scale)
        p.Tk = k.shape[2]
    else:
        B = cu_q.numel() - 1
        if max_q is None:
            max_q = int((cu_q[1:] - cu_q[:-1]).max().item()) if B > 0 else 1
        if max_k is None:
            max_k = int((cu_k[1:] - cu_k[:-1]).max().item()) if B > 0 else 1
        p = problem(B, q.shape[1], k.shape[1], max(1, max_q), q.shape[2], 64, 1, q.dtype, layout=LAYOUT_THD,
                    total_tokens=q.shape[0], scale=scale)
        p.Tk = max(1, max_k)
        p.total_keys = k.shape[0]
    p.bottom_right = int(bool(bottom_right))
    return p


def causal_fwd(q, k, v, block_size=64, window=0, bottom_right=False, cu_seqlens_q=None, cu_seqlens_k=None,
               max_seqlen_q=None, max_seqlen_k=None, scale=None, ws=None, stream=None):
    """Dense causal attention whose keys have their own lengths
    (nsa_causal_fwd): the diagonal aligned top-left (row t sees keys <= t)
    or bottom-right (keys <= t + Lk - Lq), with an optional window.
    Returns (o, lse)."""
    p = _causal_problem(q, k, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, bottom_right, scale)
    p.block_size = block_size
    o = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    _same_strides(k, v, "k and v")
    declare_strides(p, cu_seqlens_q is not None, q=q, k=k, o=o)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    L = lib()
    n = int(L.nsa_causal_fwd_workspace_size(C.byref(p)))
    if n == 0:
        raise NsaError(1, "nsa_causal_fwd_workspace_size")
    ws = workspace(n, q.device, "fwd") if ws is None else ws
    _check(L.nsa_causal_fwd(C.byref(p), int(window), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(q), _ptr(k),
                            _ptr(v), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)), "nsa_causal_fwd")
    return o, lse


def causal_bwd(q, k, v, o, dO, lse, block_size=64, window=0, bottom_right=False, cu_seqlens_q=None,
               cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None, scale=None, ws=None, stream=None,
               out=None):
    """Backward of causal_fwd (nsa_causal_bwd): returns (dq, dk, dv)."""
    p = _causal_problem(q, k, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, bottom_right, scale)
    p.block_size = block_size
    if out is None:
        dq = torch.empty(q.shape, dtype=q.dtype, device=q.device)
        dk = torch.empty(k.shape, dtype=k.dtype, device=k.device)
        dv = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    else:
        dq, dk, dv = out
    _same_strides(k, v, "k and v")
    _same_strides(o, dO, "o and dO")
    _same_strides(dk, dv, "dk and dv")
    declare_strides(p, cu_seqlens_q is not None, q=q, k=k, o=o, dq=dq, dk=dk)
    L = lib()
    n = int(L.nsa_causal_bwd_workspace_size(C.byref(p)))
    if n == 0:
        raise NsaError(1, "nsa_causal_bwd_workspace_size")
    ws = workspace(n, q.device, "bwd") if ws is None else ws
    _check(L.nsa_causal_bwd(C.byref(p), int(window), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(q), _ptr(k),
                            _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                            ws.numel(), _stream(stream)), "nsa_causal_bwd")
    return dq, dk, dv


def do_dot(o, dO, cu_seqlens=None, stream=None):
    p = problem_from(o, o, 16, 1, None, cu_seqlens)
    _same_strides(o, dO, "o and dO")
    declare_strides(p, cu_seqlens is not None, o=o)
    delta = torch.empty(o.shape[:-1], dtype=torch.float32, device=o.device)
    _check(lib().nsa_do_dot(C.byref(p), _ptr(cu_seqlens), _ptr(o), _ptr(dO), _ptr(delta),
                            _stream(stream)), "nsa_do_dot")
    return delta


def build_inverse_index(block_idx, Hq, block_size, cu_seqlens=None, max_seqlen=None,
                        stream=None):
    """Returns (offsets, rows) device int32 tensors (rows trimmed on the host)."""
    if cu_seqlens is None:
        B, Hkv, T, S = block_idx.shape
        p = problem(B, Hq, Hkv, T, 64, block_size, S, torch.bfloat16)
        ntok = B * T
    else:
        total, Hkv, S = block_idx.shape
        B = cu_seqlens.numel() - 1
        if max_seqlen is None:
            max_seqlen = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item())
        p = problem(B, Hq, Hkv, max(1, max_seqlen), 64, block_size, S, torch.bfloat16,
                    layout=LAYOUT_THD, total_tokens=total)
        ntok = total
    L = lib()
    noff = int(L.nsa_inverse_index_offsets_len(C.byref(p)))
    offsets = torch.empty(noff, dtype=torch.int32, device=block_idx.device)
    rows = torch.empty(max(1, ntok * Hkv * S), dtype=torch.int32, device=block_idx.device)
    ws = workspace(bwd_workspace_size(p), block_idx.device, "csr")
    _check(L.nsa_build_inverse_index(C.byref(p), _ptr(cu_seqlens), _ptr(block_idx), _ptr(offsets),
                                     _ptr(rows), _ptr(ws), ws.numel(), _stream(stream)),
           "nsa_build_inverse_index")
    return offsets, rows, ws


def get_error(ws, stream=None) -> int:
    out = C.c_int32(0)
    _check(lib().nsa_get_error(_ptr(ws), _stream(stream), C.byref(out)), "nsa_get_error")
    return int(out.value)


def count_pairs(block_idx, Hq, block_size, cu_seqlens=None, max_seqlen=None, stream=None) -> int:
    if cu_seqlens is None:
        B, Hkv, T, S = block_idx.shape
        p = problem(B, Hq, Hkv, T, 64, block_size, S, torch.bfloat16)
    else:
        total, Hkv, S = block_idx.shape
        B = cu_seqlens.numel() - 1
        if max_seqlen is None:
            max_seqlen = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item())
        p = problem(B, Hq, Hkv, max(1, max_seqlen), 64, block_size, S, torch.bfloat16,
                    layout=LAYOUT_THD, total_tokens=total)
    out = torch.zeros(1, dtype=torch.int64, device=block_idx.device)
    _check(lib().nsa_count_pairs(C.byref(p), _ptr(cu_seqlens), _ptr(block_idx), _ptr(out),
                                 _stream(stream)), "nsa_count_pairs")
    return int(out.item())


def debug_stall(kernel: int, wait_limit_us: int):
    """Self-test of the kernels' bounded waits (nsa_debug_stall): kernel 1
    (forward), 2 (dK/dV) or 3 (dQ) runs with its S-product issuer idle and
    every wait gives up after wait_limit_us; (0, 0) restores normal operation."""
    _check(lib().nsa_debug_stall(int(kernel), int(wait_limit_us)), "nsa_debug_stall")


def trace_enable(max_records: int):
    _check(lib().nsa_trace_enable(int(max_records)), "nsa_trace_enable")


def trace_reset():
    lib().nsa_trace_reset()


def trace_records():
    """[(kernel name, ms)] of the launches recorded since the last reset."""
    L = lib()
    out = []
    name = C.c_char_p()
    ms = C.c_float()
    for i in range(int(L.nsa_trace_count())):
        _check(L.nsa_trace_get(i, C.byref(name), C.byref(ms)), "nsa_trace_get")
        out.append((name.value.decode(), float(ms.value)))
    return out


def default_scale(D):
    return 1.0 / math.sqrt(D)


# ---------------------------------------------------------------- block selection
# The step that produces the index (include/nsa.h states the reading): block
# scores from compressed keys, then the own block and the S - 1 best complete
# blocks per index row.


def _nb(T, block_size):
    return (T + block_size - 1) // block_size


def compress_keys_mean(k, block_size, cu_seqlens=None, max_seqlen=None, stream=None):
    """kc [B, Hkv, nb, D] (k's dtype): the mean of each complete block's keys."""
    p = problem_from(k, k, block_size, 1, None, cu_seqlens, max_seqlen)
    declare_strides(p, cu_seqlens is not None, k=k)
    B = p.B
    kc = torch.empty(B, p.Hkv, _nb(p.T, block_size), p.D, dtype=k.dtype, device=k.device)
    _check(lib().nsa_compress_keys_mean(C.byref(p), _ptr(cu_seqlens), _ptr(k), _ptr(kc), _stream(stream)),
           "nsa_compress_keys_mean")
    return kc


def block_scores(q, kc, block_size, scale=None, cu_seqlens=None, max_seqlen=None, ws=None, stream=None):
    """float32 block scores, [B, Hkv, T, nb] (THD [total, Hkv, nb])."""
    p = problem_from(q, kc, block_size, 1, scale, cu_seqlens, max_seqlen)
    declare_strides(p, cu_seqlens is not None, q=q)
    nb = _nb(p.T, block_size)
    if kc.shape[2] != nb or not kc.is_contiguous():
        raise NsaError(1, "block_scores: kc must be a dense [B, Hkv, ceil(T / block_size), D] tensor")
    shape = (p.B, p.Hkv, p.T, nb) if cu_seqlens is None else (q.shape[0], p.Hkv, nb)
    scores = torch.empty(shape, dtype=torch.float32, device=q.device)
    n = int(lib().nsa_select_workspace_size(C.byref(p)))
    if n == 0:
        raise NsaError(1, "nsa_select_workspace_size")
    ws = workspace(n, q.device, "select") if ws is None else ws
    _check(lib().nsa_block_scores(C.byref(p), _ptr(cu_seqlens), _ptr(q), _ptr(kc), _ptr(scores), _ptr(ws),
                                  ws.numel(), _stream(stream)), "nsa_block_scores")
    return scores


def select_topk(scores, block_size, S, cu_seqlens=None, max_seqlen=None, stream=None):
    """int32 index rows from block scores: [B, Hkv, T, S] (THD [total, Hkv, S])."""
    if cu_seqlens is None:
        B, Hkv, T, nb = scores.shape
        p = problem(B, Hkv, Hkv, T, 32, block_size, S, torch.float32)
        shape = (B, Hkv, T, S)
    else:
        total, Hkv, nb = scores.shape
        B = cu_seqlens.numel() - 1
        if max_seqlen is None:
            max_seqlen = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()) if B > 0 else 1
        p = problem(B, Hkv, Hkv, max(1, max_seqlen), 32, block_size, S, torch.float32, layout=LAYOUT_THD,
                    total_tokens=total)
        shape = (total, Hkv, S)
    if nb != _nb(p.T, block_size) or not scores.is_contiguous():
        raise NsaError(1, "select_topk: scores must be dense with ceil(T / block_size) entries per row")
    idx = torch.empty(shape, dtype=torch.int32, device=scores.device)
    _check(lib().nsa_select_topk(C.byref(p), _ptr(cu_seqlens), _ptr(scores), _ptr(idx), _stream(stream)),
           "nsa_select_topk")
    return idx
