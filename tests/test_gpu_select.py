"""Parity of the selection step (the step that produces the index) on the GPU
with the fp64 CPU oracle, through the C ABI.

* compressed keys (mean of each complete block's keys): fp32 within fp32
  summation error, bf16 within the output's own rounding;
* block scores (compressed-attention probabilities summed over a kv
  group's heads) on the tensor cores: within the tolerance derived below;
* top-S selection from given fp32 scores: bit-exact (both sides decide on
  the same fp32 values), with ties and NaN scores;
* the whole step (GPU scores, then GPU top-S) at the headline workload's
  full size: scores against the oracle's, and every index row checked valid
  against the oracle's fp64 scores (the own block first, then complete blocks
  in decreasing score order, none left out that scores higher, up to the
  scores' tolerance), since near-ties may order differently in fp32 and fp64.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_do_gb300 import api, inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_sparse_attention_do_gb300 import build

    build.build()
    api.lib()


def _score_tol(dtype, G):
    """Max-abs tolerance of a block score (a sum of G probabilities).

    bf16 inputs: the logits are exact products summed in fp32 (relative error
    ~D * 2^-24), the exponentials ex2.approx (relative ~2^-22) and the sums
    fp32, so each probability is good to ~1e-6 relative; 1e-5 per head
    leaves a margin of 10.  fp32 inputs run in split precision (about 2^-16 of
    |q||kc| per logit, i.e. ~1e-4 on logits of size ~10 with D = 128), so
    1e-4 per head."""
    return (1e-5 if dtype == torch.bfloat16 else 1e-4) * max(G, 1)


def _scores_gpu(q, kc, bs, cu=None, max_seqlen=None):
    qd = q.to(DEV)
    kd = kc.to(DEV)
    cud = None if cu is None else cu.to(DEV)
    sc = api.block_scores(qd, kd, bs, cu_seqlens=cud, max_seqlen=max_seqlen)
    ws = api.workspace(256, DEV, "select")
    torch.cuda.synchronize()
    err = C_err(ws)
    assert err == 0, f"device error {err}"
    return sc.cpu()


def C_err(ws):
    import ctypes as C

    out = C.c_int32(-1)
    assert api.lib().nsa_get_error(api._ptr(ws), api._stream(), C.byref(out)) == 0
    return out.value


# ------------------------------------------------------------ compressed keys
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T,bs,D", [(200, 16, 64), (130, 64, 128), (37, 32, 32)])
def test_compress_mean(dtype, T, bs, D):
    B, Hkv = 2, 3
    _, k, _, _ = inputs.make_qkv_do(B, Hkv, Hkv, T, D, dtype=dtype, seed=21)
    got = api.compress_keys_mean(k.to(DEV), bs).cpu()
    ref = oracle.compress_mean(k, bs)
    assert got.shape == ref.shape and got.dtype == dtype
    err = np.abs(got.double().numpy() - ref)
    if dtype == torch.bfloat16:
        err = err - 2.0 ** -8 * np.abs(ref)  # the output's own rounding
    assert err.max() <= 1e-6, err.max()


def test_compress_mean_packed_and_strided():
    bs, Hq, Hkv, D = 16, 4, 2, 64
    lens = [70, 5, 33, 128]
    cu = inputs.cu_seqlens_from_lengths(lens)
    total = sum(lens)
    # k as a view of a packed [total, Hq + 2 Hkv, D] qkv tensor
    g = torch.Generator().manual_seed(22)
    qkv = torch.randn(total, Hq + 2 * Hkv, D, generator=g).to(torch.bfloat16)
    k = qkv[:, Hq : Hq + Hkv]
    got = api.compress_keys_mean(qkv.to(DEV)[:, Hq : Hq + Hkv], bs, cu_seqlens=cu.to(DEV)).cpu()
    ref = oracle.compress_mean(k, bs, cu_seqlens=cu)
    err = np.abs(got.double().numpy() - ref) - 2.0 ** -8 * np.abs(ref)
    assert err.max() <= 1e-6, err.max()


# --------------------------------------------------------------- block scores
SCORE_CASES = [
    # B, Hq, Hkv, T, D, bs, dtype
    (2, 4, 2, 200, 64, 16, torch.bfloat16),    # G = 2, ragged tail
    (1, 16, 1, 300, 128, 64, torch.bfloat16),  # G = 16
    (1, 6, 2, 130, 32, 32, torch.float32),     # D = 32 (padded), split precision
    (2, 4, 2, 150, 128, 32, torch.float32),    # fp32 D = 128
    (1, 128, 1, 70, 64, 16, torch.bfloat16),   # G = 128: one token per tile
    (1, 3, 3, 4200, 64, 16, torch.bfloat16),   # 263 blocks: S recomputed in pass 2
    (1, 2, 1, 10, 64, 16, torch.float32),      # T < block size: no complete block
    (1, 4, 2, 150, 32, 16, torch.bfloat16),    # bf16 D = 32: per-thread copies, not TMA
]


@pytest.mark.parametrize("B,Hq,Hkv,T,D,bs,dtype", SCORE_CASES)
def test_block_scores(B, Hq, Hkv, T, D, bs, dtype):
    q, _, _, _ = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=dtype, seed=23)
    nb = (T + bs - 1) // bs
    kc = inputs.make_compressed_keys(B, Hkv, nb, D, dtype=dtype, seed=24)
    got = _scores_gpu(q, kc, bs)
    ref = oracle.block_scores(q, kc, bs)
    assert got.shape == ref.shape
    err = float(np.max(np.abs(got.double().numpy() - ref)))
    assert err <= _score_tol(dtype, Hq // Hkv), err
    # blocks not complete at a row score exactly 0
    t = np.arange(T)[:, None]
    j = np.arange(nb)[None, :]
    assert np.all(got.numpy()[..., (j + 1) * bs - 1 > t] == 0.0)


@pytest.mark.parametrize("Hq,Hkv,D,bs", [(8, 2, 64, 32), (32, 2, 128, 64)])
def test_block_scores_packed_sequences(Hq, Hkv, D, bs):
    lens = [100, 7, 260, 33]
    cu = inputs.cu_seqlens_from_lengths(lens)
    total = sum(lens)
    q, _, _, _ = inputs.make_qkv_do(1, Hq, Hkv, total, D, dtype=torch.bfloat16, seed=25, layout="thd")
    nb = (max(lens) + bs - 1) // bs
    kc = inputs.make_compressed_keys(len(lens), Hkv, nb, D, dtype=torch.bfloat16, seed=26)
    got = _scores_gpu(q, kc, bs, cu=cu)
    ref = oracle.block_scores(q, kc, bs, cu_seqlens=cu)
    err = float(np.max(np.abs(got.double().numpy() - ref)))
    assert err <= _score_tol(torch.bfloat16, Hq // Hkv), err


# ------------------------------------------------------------------- top-S
@pytest.mark.parametrize("S", [1, 4, 16, 40])
@pytest.mark.parametrize("levels,nan_frac", [(0, 0.0), (4, 0.05)])
def test_select_topk_bit_exact(S, levels, nan_frac):
    B, Hkv, T, bs = 2, 3, 300, 16
    nb = (T + bs - 1) // bs
    sc = inputs.make_block_scores((B, Hkv, T, nb), seed=27, levels=levels, nan_frac=nan_frac)
    got = api.select_topk(sc.to(DEV), bs, S).cpu().numpy()
    ref = oracle.select_topk(sc, bs, S)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("T", [900, 3000])  # rows of up to 57 and 188 blocks
def test_select_topk_row_lengths(T):
    B, Hkv, bs, S = 1, 2, 16, 16
    nb = (T + bs - 1) // bs
    sc = inputs.make_block_scores((B, Hkv, T, nb), seed=31, levels=8, nan_frac=0.02)
    got = api.select_topk(sc.to(DEV), bs, S).cpu().numpy()
    ref = oracle.select_topk(sc, bs, S)
    np.testing.assert_array_equal(got, ref)


def test_select_topk_packed_and_long_rows():
    lens = [1000, 3, 64, 4200]
    Hkv, bs, S = 2, 16, 24  # up to 263 blocks a row
    cu = inputs.cu_seqlens_from_lengths(lens)
    nb = (max(lens) + bs - 1) // bs
    sc = inputs.make_block_scores((sum(lens), Hkv, nb), seed=28, levels=16, nan_frac=0.01)
    got = api.select_topk(sc.to(DEV), bs, S, cu_seqlens=cu.to(DEV)).cpu().numpy()
    ref = oracle.select_topk(sc, bs, S, cu_seqlens=cu)
    np.testing.assert_array_equal(got, ref)


# ------------------------------------------------- the whole step, full size
def _check_selection(idx, ref, bs, S, tol):
    """Every row: own block first, then distinct complete blocks in
    decreasing (fp64) score order, none left out that scores higher, up to
    tol; -1 after them."""
    B, Hkv, T, nb = ref.shape
    for b in range(B):
        for g in range(Hkv):
            for t in range(T):
                row = idx[b, g, t]
                own, nc = t // bs, (t + 1) // bs
                assert row[0] == own
                cand = [j for j in range(nc) if j != own]
                n = min(S - 1, len(cand))
                picks = row[1 : 1 + n]
                assert np.all(row[1 + n :] == -1)
                assert len(set(picks.tolist())) == n and all(0 <= j < nc and j != own for j in picks)
                sc = ref[b, g, t]
                if n:
                    assert np.all(np.diff(sc[picks]) <= tol)
                    rest = np.setdiff1d(np.array(cand, dtype=np.int64), picks)
                    if rest.size:
                        assert sc[picks].min() >= sc[rest].max() - tol


def test_selection_step_headline_workload():
    """B=1 Hq=32 Hkv=2 T=8192 D=128, 64-key blocks, S=16, bf16."""
    B, Hq, Hkv, T, D, bs, S = 1, 32, 2, 8192, 128, 64, 16
    q, k, _, _ = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.bfloat16, seed=29)
    nb = T // bs
    kc = inputs.make_compressed_keys(B, Hkv, nb, D, dtype=torch.bfloat16, seed=30)
    got = _scores_gpu(q, kc, bs)
    idx = api.select_topk(got.to(DEV), bs, S).cpu().numpy()
    ref = oracle.block_scores(q, kc, bs)
    tol = _score_tol(torch.bfloat16, Hq // Hkv)
    err = float(np.max(np.abs(got.double().numpy() - ref)))
    assert err <= tol, err
    _check_selection(idx, ref, bs, S, 2 * tol)
    # the index feeds the selection backward's validation unchanged
    assert oracle.validate_index(torch.from_numpy(idx), bs) == 0
