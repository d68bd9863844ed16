"""The seeded generators: determinism and the structure of the block index."""
import numpy as np
import torch

from block_sparse_attention_do_gb300 import inputs


def test_qkv_deterministic_and_rounded():
    a = inputs.make_qkv_do(1, 4, 2, 16, 8, dtype=torch.bfloat16, seed=3)
    b = inputs.make_qkv_do(1, 4, 2, 16, 8, dtype=torch.bfloat16, seed=3)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and torch.equal(x, y)
    c = inputs.make_qkv_do(1, 4, 2, 16, 8, seed=4)
    assert not torch.equal(a[0].float(), c[0])


def test_block_idx_structure():
    B, Hkv, T, bs, S = 2, 3, 300, 16, 5
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=0).numpy()
    assert idx.shape == (B, Hkv, T, S) and idx.dtype == np.int32
    assert np.array_equal(idx, inputs.make_block_idx(B, Hkv, T, bs, S, seed=0).numpy())
    for b in range(B):
        for g in range(Hkv):
            for t in range(T):
                row = idx[b, g, t]
                own = t // bs
                assert row[0] == own
                rest = row[1:]
                valid = rest[rest >= 0]
                assert len(valid) == min(S - 1, own)
                assert np.all(np.diff(valid) > 0) and np.all(valid < own)
                assert np.all(rest[len(valid):] == -1)


def test_block_idx_is_roughly_uniform():
    T, bs, S = 64 * 64, 64, 16
    idx = inputs.make_block_idx(1, 1, T, bs, S, seed=0).numpy()[0, 0]
    last = idx[T - bs:, 1:]  # rows of block 63 pick 15 of 63 earlier blocks
    counts = np.bincount(last.ravel(), minlength=63)[:63]
    expect = bs * 15 / 63
    assert counts.min() > 0.4 * expect and counts.max() < 1.8 * expect


def test_varlen_lengths_and_idx():
    lengths = inputs.make_varlen_lengths(8, 128, 4096, seed=0)
    assert len(lengths) == 8 and all(128 <= L <= 4096 for L in lengths)
    cu = inputs.cu_seqlens_from_lengths(lengths)
    assert cu[0] == 0 and int(cu[-1]) == sum(lengths)
    idx = inputs.make_varlen_block_idx(lengths[:2], 2, 64, 16)
    assert idx.shape == (sum(lengths[:2]), 2, 16)
    L0 = lengths[0]
    assert np.array_equal(idx[:L0, 0, 0].numpy(), np.arange(L0) // 64)
    assert np.array_equal(idx[L0:, 1, 0].numpy(), np.arange(lengths[1]) // 64)


def test_dense_idx():
    idx = inputs.make_dense_block_idx(1, 1, 10, 4).numpy()[0, 0]
    assert idx.shape == (10, 3)
    assert list(idx[0]) == [0, -1, -1] and list(idx[9]) == [0, 1, 2]
