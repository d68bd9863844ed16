"""Seeded synthetic inputs for NSA block-selection attention.

This module is shared by the oracle tests, the CUDA parity tests and the
benchmark.  It holds random-number plumbing only and none of the attention
arithmetic: it draws q, k, v, dO, the per-token block-selection index and the
packed variable-length sequence lengths.

Recipe (the gradcheck-gate page, ``test_kernel_backward.py``, ``run_one``):
``torch.manual_seed(seed)`` then standard-normal q, k, v and dO with shapes
[B, Hq, T, D] / [B, Hkv, T, D].  The page draws them on the GPU; here they are
drawn on the CPU in fp32 (so that CPU and GPU sides see identical values) and
then rounded to the compute dtype.  The block index comes from
``make_block_idx(B, Hkv, T, block_size, S, seed)``, which the page imports but
does not print; the reading taken here is:

* slot 0 holds the token's own causal block ``t // block_size``;
* slots 1 .. holds ``min(S - 1, t // block_size)`` distinct earlier blocks
  drawn uniformly without replacement, in ascending order;
* remaining slots hold -1 (padding).
"""
from __future__ import annotations

import numpy as np
import torch

__all__ = [
    "make_qkv_do",
    "make_block_idx",
    "make_dense_block_idx",
    "make_varlen_lengths",
    "make_varlen_block_idx",
    "cu_seqlens_from_lengths",
    "round_to_dtype",
    "make_compressed_keys",
    "make_block_scores",
]


def round_to_dtype(x: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    """Round an fp32 CPU tensor to ``dtype`` (round-to-nearest-even)."""
    return x.to(dtype)


def make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.float32, seed=0, layout="bhtd"):
    """Return (q, k, v, dO) CPU tensors in ``dtype``.

    layout "bhtd": q/dO [B, Hq, T, D], k/v [B, Hkv, T, D].
    layout "thd":  B is ignored, T is the packed token total: q/dO [T, Hq, D],
    k/v [T, Hkv, D].
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    if layout == "bhtd":
        qs, ks = (B, Hq, T, D), (B, Hkv, T, D)
    elif layout == "thd":
        qs, ks = (T, Hq, D), (T, Hkv, D)
    else:
        raise ValueError(layout)
    q = torch.randn(qs, generator=g, dtype=torch.float32)
    k = torch.randn(ks, generator=g, dtype=torch.float32)
    v = torch.randn(ks, generator=g, dtype=torch.float32)
    do = torch.randn(qs, generator=g, dtype=torch.float32)
    return tuple(round_to_dtype(x, dtype) for x in (q, k, v, do))


def _draw_rows(rng: np.random.Generator, L: int, bs: int, S: int) -> np.ndarray:
    """Selection rows for one (sequence, kv head): int32 [L, S]."""
    nb = (L + bs - 1) // bs
    out = np.full((L, S), -1, dtype=np.int32)
    t = np.arange(L)
    own = t // bs
    out[:, 0] = own
    if S == 1 or nb == 1:
        # every row already holds its own block; still advance the stream the
        # same way for every shape so seeds stay comparable
        rng.random((L, max(nb, 1)))
        return out
    keys = rng.random((L, nb))
    # only strictly earlier blocks are candidates
    cand = np.arange(nb)[None, :] < own[:, None]
    keys = np.where(cand, keys, np.inf)
    order = np.argsort(keys, axis=1, kind="stable")[:, : S - 1]
    if order.shape[1] < S - 1:  # fewer blocks than slots: pad the candidate list
        order = np.pad(order, ((0, 0), (0, S - 1 - order.shape[1])), constant_values=0)
    take = np.minimum(S - 1, own)  # how many earlier blocks each row gets
    picked = np.where(np.arange(S - 1)[None, :] < take[:, None], order, np.iinfo(np.int32).max)
    picked = np.sort(picked, axis=1)
    picked = np.where(picked == np.iinfo(np.int32).max, -1, picked)
    out[:, 1:] = picked.astype(np.int32)
    return out


def make_block_idx(B, Hkv, T, bs, S, seed=0) -> torch.Tensor:
    """int32 [B, Hkv, T, S] selection index (see module docstring)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = np.empty((B, Hkv, T, S), dtype=np.int32)
    for b in range(B):
        for g in range(Hkv):
            out[b, g] = _draw_rows(rng, T, bs, S)
    return torch.from_numpy(out)


def make_dense_block_idx(B, Hkv, T, bs) -> torch.Tensor:
    """int32 [B, Hkv, T, nb]: every row selects all of its blocks 0..t//bs."""
    nb = (T + bs - 1) // bs
    t = np.arange(T)[:, None]
    j = np.arange(nb)[None, :]
    row = np.where(j <= t // bs, j, -1).astype(np.int32)
    return torch.from_numpy(np.broadcast_to(row, (B, Hkv, T, nb)).copy())


def make_varlen_lengths(n_seqs, lo, hi, seed=0) -> list[int]:
    """Sequence lengths drawn uniformly from the integers [lo, hi]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return [int(x) for x in rng.integers(lo, hi + 1, size=n_seqs)]


def cu_seqlens_from_lengths(lengths) -> torch.Tensor:
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return torch.from_numpy(cu)


def make_varlen_block_idx(lengths, Hkv, bs, S, seed=0) -> torch.Tensor:
    """int32 [total, Hkv, S] with sequence-local block ids."""
    rng = np.random.Generator(np.random.PCG64(seed))
    total = int(sum(lengths))
    out = np.empty((total, Hkv, S), dtype=np.int32)
    off = 0
    for L in lengths:
        for g in range(Hkv):
            out[off : off + L, g, :] = _draw_rows(rng, L, bs, S)
        off += L
    return torch.from_numpy(out)


def make_compressed_keys(B, Hkv, nb, D, dtype=torch.float32, seed=0) -> torch.Tensor:
    """[B, Hkv, nb, D] CPU tensor in ``dtype``: standard normal draws standing
    in for one compressed key per key block."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return round_to_dtype(torch.randn((B, Hkv, nb, D), generator=g, dtype=torch.float32), dtype)


def make_block_scores(shape, seed=0, levels=0, nan_frac=0.0) -> torch.Tensor:
    """fp32 CPU tensor of block scores: uniform in [0, 1), or (levels > 0)
    one of ``levels`` evenly spaced values so that ties are common; a
    fraction ``nan_frac`` of the entries is NaN."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    if levels > 0:
        x = torch.randint(0, levels, shape, generator=g).float() / levels
    else:
        x = torch.rand(shape, generator=g, dtype=torch.float32)
    if nan_frac > 0:
        x[torch.rand(shape, generator=g) < nan_frac] = float("nan")
    return x
