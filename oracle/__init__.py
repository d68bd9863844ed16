"""Python loader for the fp64 CPU oracle (``nsa_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the smoke check and by
the benchmark's CPU-baseline leg.  The product library never imports it.

Every wrapper takes numpy-convertible arrays (torch CPU tensors work), turns
the floating-point ones into contiguous fp64 and returns fp64 numpy arrays.
Layouts follow the C file: fixed length [B, H, T, D] when ``cu_seqlens`` is
None, packed [total, H, D] otherwise.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nsa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_i64 = C.c_int64
_dbl = C.c_double
_ptr = C.c_void_p


def build(force: bool = False) -> str:
    """Compile liboracle.so with the host C compiler (gcc/cc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cc = os.environ.get("CC", "gcc")
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call([cc, "-O2", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB)
        L.oracle_validate_index.restype = C.c_int
        L.oracle_validate_index.argtypes = [_i64] * 5 + [_ptr, _ptr]
        common = [_i64] * 7 + [_dbl, _ptr]
        L.oracle_sel_fwd_w.restype = None
        L.oracle_sel_fwd_w.argtypes = common + [_ptr] * 6 + [_i64]
        L.oracle_sel_bwd_w.restype = None
        L.oracle_sel_bwd_w.argtypes = common + [_ptr] * 11 + [_i64]
        L.oracle_sel_fwd_s.restype = None
        L.oracle_sel_fwd_s.argtypes = common + [_ptr] * 6 + [_i64, _ptr]
        L.oracle_sel_bwd_s.restype = None
        L.oracle_sel_bwd_s.argtypes = common + [_ptr] * 11 + [_i64, _ptr, _ptr]
        L.oracle_inverse_index.restype = None
        L.oracle_inverse_index.argtypes = [_i64] * 5 + [_ptr, _ptr, _i64, _ptr, _ptr]
        L.oracle_do_dot.restype = None
        L.oracle_do_dot.argtypes = [_i64] * 4 + [_ptr] * 4
        L.oracle_count_pairs_w.restype = _i64
        L.oracle_count_pairs_w.argtypes = [_i64] * 6 + [_ptr, _ptr, _i64]
        L.oracle_sel_rows_w.restype = None
        L.oracle_sel_rows_w.argtypes = common + [_ptr] * 5 + [_i64] + [_ptr] * 6 + [_i64]
        L.oracle_sel_keys_w.restype = None
        L.oracle_sel_keys_w.argtypes = common + [_ptr] * 5 + [_i64] + [_ptr] * 5 + [_i64]
        L.oracle_sel_blocks_w.restype = None
        L.oracle_sel_blocks_w.argtypes = common + [_ptr] * 5 + [_i64] + [_ptr] * 5 + [_i64]
        L.oracle_compress_mean.restype = None
        L.oracle_compress_mean.argtypes = [_i64] * 6 + [_ptr] * 3
        L.oracle_block_scores.restype = None
        L.oracle_block_scores.argtypes = [_i64] * 7 + [_dbl] + [_ptr] * 4
        L.oracle_select_topk.restype = None
        L.oracle_select_topk.argtypes = [_i64] * 6 + [_ptr] * 3
        _lib = L
    return _lib


def _f64(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _i32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _shape(q, k, idx, cu_seqlens):
    """(B, Hq, Hkv, T, D, S) from the tensors' shapes."""
    if cu_seqlens is None:
        B, Hq, T, D = q.shape
        Hkv = k.shape[1]
        S = idx.shape[3]
    else:
        T, Hq, D = q.shape  # T = packed total
        Hkv = k.shape[1]
        S = idx.shape[2]
        B = len(cu_seqlens) - 1
    return B, Hq, Hkv, T, D, S


def sel_fwd(q, k, v, idx, bs, scale=None, cu_seqlens=None, window=0, sinks=None):
    """Returns (O, LSE) in fp64.  window > 0: keys k with t - k < window only.
    sinks: one logit per query head in every row's softmax denominator."""
    q, k, v, idx, cu = _f64(q), _f64(k), _f64(v), _i32(idx), _i32(cu_seqlens)
    B, Hq, Hkv, T, D, S = _shape(q, k, idx, cu)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    sk = None if sinks is None else _f64(sinks)
    o = np.zeros_like(q)
    lse = np.zeros(q.shape[:-1], dtype=np.float64)
    lib().oracle_sel_fwd_s(B, Hq, Hkv, T, D, bs, S, scale, _p(cu), _p(q), _p(k), _p(v), _p(idx),
                           _p(o), _p(lse), int(window), _p(sk))
    return o, lse


def sel_bwd(q, k, v, idx, dO, bs, scale=None, cu_seqlens=None, want_dsum=False, window=0, sinks=None):
    """Returns dict with dq, dk, dv, o, lse (and dsum = row sums of dS; with
    sinks, dsinks = the gradient of the sink logits)."""
    q, k, v, dO, idx, cu = _f64(q), _f64(k), _f64(v), _f64(dO), _i32(idx), _i32(cu_seqlens)
    B, Hq, Hkv, T, D, S = _shape(q, k, idx, cu)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    sk = None if sinks is None else _f64(sinks)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    o = np.zeros_like(q)
    lse = np.zeros(q.shape[:-1], dtype=np.float64)
    dsum = np.zeros(q.shape[:-1], dtype=np.float64) if want_dsum else None
    dsk = None if sk is None else np.zeros_like(sk)
    lib().oracle_sel_bwd_s(B, Hq, Hkv, T, D, bs, S, scale, _p(cu), _p(q), _p(k), _p(v), _p(idx),
                           _p(dO), _p(dq), _p(dk), _p(dv), _p(o), _p(lse), _p(dsum), int(window), _p(sk),
                           _p(dsk))
    out = dict(dq=dq, dk=dk, dv=dv, o=o, lse=lse)
    if want_dsum:
        out["dsum"] = dsum
    if dsk is not None:
        out["dsinks"] = dsk
    return out


def validate_index(idx, bs, cu_seqlens=None, T=None):
    """0 when the index is valid, 3 (bad index) otherwise."""
    idx, cu = _i32(idx), _i32(cu_seqlens)
    if cu is None:
        B, Hkv, T, S = idx.shape
    else:
        T, Hkv, S = idx.shape
        B = len(cu) - 1
    return int(lib().oracle_validate_index(B, Hkv, T, bs, S, _p(cu), _p(idx)))


def inverse_index(idx, bs, cu_seqlens=None):
    """Returns (offsets int32 [B*Hkv*nbmax + 1], rows int32 [nnz], nbmax)."""
    idx, cu = _i32(idx), _i32(cu_seqlens)
    if cu is None:
        B, Hkv, T, S = idx.shape
        maxlen = T
    else:
        T, Hkv, S = idx.shape
        B = len(cu) - 1
        maxlen = int(np.max(np.diff(cu))) if B > 0 else 0
    nbmax = (maxlen + bs - 1) // bs
    offsets = np.zeros(B * Hkv * nbmax + 1, dtype=np.int32)
    rows = np.zeros(max(1, idx.size), dtype=np.int32)
    lib().oracle_inverse_index(B, Hkv, T, bs, S, _p(cu), _p(idx), nbmax, _p(offsets), _p(rows))
    return offsets, rows[: offsets[-1]].copy(), nbmax


def do_dot(o, dO, cu_seqlens=None):
    o, dO, cu = _f64(o), _f64(dO), _i32(cu_seqlens)
    if cu is None:
        B, H, T, D = o.shape
    else:
        T, H, D = o.shape
        B = len(cu) - 1
    out = np.zeros(o.shape[:-1], dtype=np.float64)
    lib().oracle_do_dot(B, H, T, D, _p(cu), _p(o), _p(dO), _p(out))
    return out


def count_pairs(idx, Hq, bs, cu_seqlens=None, window=0):
    idx, cu = _i32(idx), _i32(cu_seqlens)
    if cu is None:
        B, Hkv, T, S = idx.shape
    else:
        T, Hkv, S = idx.shape
        B = len(cu) - 1
    return int(lib().oracle_count_pairs_w(B, Hq, Hkv, T, bs, S, _p(cu), _p(idx), int(window)))


def sel_rows(q, k, v, idx, dO, bs, rows, scale=None, cu_seqlens=None, window=0):
    """rows: int array [n, 3] of (b, h, t).  Returns (o [n,D], lse [n], dq [n,D])."""
    q, k, v, dO, idx, cu = _f64(q), _f64(k), _f64(v), _f64(dO), _i32(idx), _i32(cu_seqlens)
    B, Hq, Hkv, T, D, S = _shape(q, k, idx, cu)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    rb, rh, rt = (np.ascontiguousarray(rows[:, i]) for i in range(3))
    n = rows.shape[0]
    o, lse, dq = np.zeros((n, D)), np.zeros(n), np.zeros((n, D))
    lib().oracle_sel_rows_w(B, Hq, Hkv, T, D, bs, S, scale, _p(cu), _p(q), _p(k), _p(v), _p(idx),
                            _p(dO), n, _p(rb), _p(rh), _p(rt), _p(o), _p(lse), _p(dq), int(window))
    return o, lse, dq


def sel_keys(q, k, v, idx, dO, bs, keys, scale=None, cu_seqlens=None, window=0):
    """keys: int array [n, 3] of (b, g, key).  Returns (dk [n,D], dv [n,D])."""
    q, k, v, dO, idx, cu = _f64(q), _f64(k), _f64(v), _f64(dO), _i32(idx), _i32(cu_seqlens)
    B, Hq, Hkv, T, D, S = _shape(q, k, idx, cu)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    keys = np.ascontiguousarray(np.asarray(keys, dtype=np.int64).reshape(-1, 3))
    kb, kg, kk = (np.ascontiguousarray(keys[:, i]) for i in range(3))
    n = keys.shape[0]
    dk, dv = np.zeros((n, D)), np.zeros((n, D))
    lib().oracle_sel_keys_w(B, Hq, Hkv, T, D, bs, S, scale, _p(cu), _p(q), _p(k), _p(v), _p(idx),
                            _p(dO), n, _p(kb), _p(kg), _p(kk), _p(dk), _p(dv), int(window))
    return dk, dv


def sel_blocks(q, k, v, idx, dO, bs, blocks, scale=None, cu_seqlens=None, window=0):
    """blocks: int array [n, 3] of (b, g, j).  Returns (dk [n,bs,D], dv [n,bs,D]):
    dK and dV of the keys j*bs .. j*bs+bs-1 (zero past the sequence's end)."""
    q, k, v, dO, idx, cu = _f64(q), _f64(k), _f64(v), _f64(dO), _i32(idx), _i32(cu_seqlens)
    B, Hq, Hkv, T, D, S = _shape(q, k, idx, cu)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    blocks = np.ascontiguousarray(np.asarray(blocks, dtype=np.int64).reshape(-1, 3))
    nb = -(-T // bs) if cu is None else -(-int(np.max(np.diff(cu))) // bs)
    if blocks.size and (blocks.min() < 0 or blocks[:, 0].max() >= B or blocks[:, 1].max() >= Hkv
                        or blocks[:, 2].max() >= nb):
        raise ValueError("sel_blocks: (b, g, j) out of range")
    jb, jg, jj = (np.ascontiguousarray(blocks[:, i]) for i in range(3))
    n = blocks.shape[0]
    dk, dv = np.zeros((n, bs, D)), np.zeros((n, bs, D))
    lib().oracle_sel_blocks_w(B, Hq, Hkv, T, D, bs, S, scale, _p(cu), _p(q), _p(k), _p(v), _p(idx),
                              _p(dO), n, _p(jb), _p(jg), _p(jj), _p(dk), _p(dv), int(window))
    return dk, dv


def causal(q, k, v, dO=None, scale=None, cu_seqlens_q=None, cu_seqlens_k=None, window=0,
           bottom_right=False):
    """Dense causal attention with separate query and key lengths: row t of a
    sequence with Lq queries and Lk keys attends keys k <= c_t (c_t = t, or
    t + Lk - Lq with bottom_right), k < Lk, and c_t - k < window when
    window > 0.  Fixed length: q [B,Hq,Tq,D], k/v [B,Hkv,Tk,D]; packed:
    q [total_q,Hq,D], k/v [total_k,Hkv,D] with cu_seqlens_q / cu_seqlens_k.
    Returns dict(o, lse) and, with dO, dq, dk, dv (fp64)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    dOa = None if dO is None else _f64(dO)
    cuq, cuk = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    if (cuq is None) != (cuk is None):
        raise ValueError("give both cu_seqlens or neither")
    if cuq is None:
        B, Hq, Tq, D = q.shape
        Hkv, Tk = k.shape[1], k.shape[2]
    else:
        B = len(cuq) - 1
        Tq, Hq, D = q.shape
        Tk, Hkv = k.shape[0], k.shape[1]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    L = lib()
    if not hasattr(L, "_causal_set"):
        L.oracle_causal.restype = None
        L.oracle_causal.argtypes = [_i64] * 6 + [_dbl, _ptr, _ptr, _i64, _i64] + [_ptr] * 9
        L._causal_set = True
    o = np.zeros_like(q)
    lse = np.zeros(q.shape[:-1], dtype=np.float64)
    out = dict(o=o, lse=lse)
    dq = dk = dv = None
    if dOa is not None:
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        out.update(dq=dq, dk=dk, dv=dv)
    L.oracle_causal(B, Hq, Hkv, Tq, Tk, D, scale, _p(cuq), _p(cuk), int(window), int(bool(bottom_right)),
                    _p(q), _p(k), _p(v), _p(dOa), _p(o), _p(lse), _p(dq), _p(dk), _p(dv))
    return out


# ---------------------------------------------------------------- block selection
# The step that produces idx (reading in nsa_oracle.c): compressed keys (mean
# pooling stand-in), block scores = compressed-attention probabilities summed
# over a kv group's heads, and the top-S selection with the own block first.


def _nb(T, bs, cu):
    maxlen = T if cu is None else (int(np.max(np.diff(cu))) if len(cu) > 1 else 0)
    return (maxlen + bs - 1) // bs


def compress_mean(k, bs, cu_seqlens=None, T=None):
    """kc [B, Hkv, nb, D] fp64: the mean of each complete block's keys (zero
    rows elsewhere).  THD: k [total, Hkv, D]; T (optional) fixes nb's length."""
    k, cu = _f64(k), _i32(cu_seqlens)
    if cu is None:
        B, Hkv, Tt, D = k.shape
    else:
        Tt, Hkv, D = k.shape
        B = len(cu) - 1
    if cu is None:
        nb = (Tt + bs - 1) // bs
    else:  # the longest sequence's blocks, or ceil(T / bs) for a given length bound T
        nb = _nb(None, bs, cu) if T is None else (T + bs - 1) // bs
    kc = np.zeros((B, Hkv, nb, D), dtype=np.float64)
    lib().oracle_compress_mean(B, Hkv, Tt, D, bs, nb, _p(cu), _p(k), _p(kc))
    return kc


def block_scores(q, kc, bs, scale=None, cu_seqlens=None):
    """scores fp64, [B, Hkv, T, nb] (THD [total, Hkv, nb]), from q and kc [B, Hkv, nb, D]."""
    q, kc, cu = _f64(q), _f64(kc), _i32(cu_seqlens)
    B_, Hkv, nb, D = kc.shape
    if cu is None:
        B, Hq, T, _ = q.shape
        shape = (B, Hkv, T, nb)
    else:
        T, Hq, _ = q.shape
        B = len(cu) - 1
        shape = (T, Hkv, nb)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    out = np.zeros(shape, dtype=np.float64)
    lib().oracle_block_scores(B, Hq, Hkv, T, D, bs, nb, scale, _p(cu), _p(q), _p(kc), _p(out))
    return out


def select_topk(scores, bs, S, cu_seqlens=None):
    """idx int32 [B, Hkv, T, S] (THD [total, Hkv, S]) from scores (any float
    dtype; an fp32 input is compared exactly as fp32 since fp32 -> fp64 is exact)."""
    sc, cu = _f64(scores), _i32(cu_seqlens)
    if cu is None:
        B, Hkv, T, nb = sc.shape
        shape = (B, Hkv, T, S)
    else:
        T, Hkv, nb = sc.shape
        B = len(cu) - 1
        shape = (T, Hkv, S)
    idx = np.full(shape, -1, dtype=np.int32)
    lib().oracle_select_topk(B, Hkv, T, bs, S, nb, _p(cu), _p(sc), _p(idx))
    return idx
