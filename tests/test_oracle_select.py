"""Pins for the oracle's block-selection step (the step that produces idx).

The pages take the index as given, so the reading is the plainest one of
NSA's selection (stated in full in ``oracle/nsa_oracle.c``): block j is
complete at row t when (j + 1) bs - 1 <= t; a row's block scores are the
softmax over its complete blocks of scale <q, kc_j>, summed over the G query
heads of its kv head; idx is the row's own block and then the S - 1
best-scoring complete blocks (ties: smaller j first).

Each pin checks the oracle against something other than itself:

* the compressed keys against torch's mean over each block's keys;
* the scores against the oracle's dense causal attention (itself pinned to
  torch's causal SDPA bias) over the sequence of compressed keys, read out
  through one-hot values: the rows at a block's last key see blocks 0..m
  (top-left causal), the other rows see blocks 0..m-1 (bottom-right with one
  key fewer) -- a wrong completeness rule, a missing head sum, a wrong
  scale or GQA mapping fails it;
* closed forms (one complete block gives G; two give a sigmoid), the row sum
  G, zeros past the complete blocks, invariance to a shift common to every
  compressed key;
* the top-S selection against Python's sort by (-score, j), with ties and
  NaN scores, fixed length and packed sequences, and its limits (S = 1, S
  above the complete block count); every selected index passes the oracle's
  own index validation.
"""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64)


@pytest.mark.parametrize("T,bs", [(40, 8), (37, 4), (16, 16), (15, 16)])
def test_compress_mean_is_the_block_average(T, bs):
    B, Hkv, D = 2, 3, 8
    k = _rand((B, Hkv, T, D), 1)
    kc = oracle.compress_mean(k, bs)
    nb, nc = (T + bs - 1) // bs, T // bs
    assert kc.shape == (B, Hkv, nb, D)
    want = k[:, :, : nc * bs].reshape(B, Hkv, nc, bs, D).mean(dim=3).numpy()
    np.testing.assert_allclose(kc[:, :, :nc], want, rtol=0, atol=1e-14)
    assert np.all(kc[:, :, nc:] == 0.0)


def test_compress_mean_packed_sequences():
    bs, Hkv, D = 4, 2, 8
    lens = [9, 4, 3, 12]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    k = _rand((int(cu[-1]), Hkv, D), 2)
    kc = oracle.compress_mean(k, bs, cu_seqlens=cu)
    nb = (max(lens) + bs - 1) // bs
    assert kc.shape == (len(lens), Hkv, nb, D)
    for b, L in enumerate(lens):
        seq = k[cu[b] : cu[b + 1]].permute(1, 0, 2)  # [Hkv, L, D]
        nc = L // bs
        if nc:
            want = seq[:, : nc * bs].reshape(Hkv, nc, bs, D).mean(dim=2).numpy()
            np.testing.assert_allclose(kc[b, :, :nc], want, rtol=0, atol=1e-14)
        assert np.all(kc[b, :, nc:] == 0.0)


def _scores_via_causal_attention(q, kc, bs, scale):
    """Block scores rebuilt from the oracle's dense causal attention over the
    compressed keys, one query offset within the block at a time."""
    B, Hq, T, D = q.shape
    Hkv, nb = kc.shape[1], kc.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hkv, T, nb))
    for o in range(bs):
        rows = np.arange(o, T, bs)  # t = m bs + o, m = 0 .. M-1
        M = len(rows)
        last = o == bs - 1
        Lk = M if last else M - 1  # keys 0..m (top-left) or 0..m-1 (bottom-right)
        if M == 0 or Lk <= 0:
            continue
        assert Lk <= D, "one-hot values need D >= the compressed key count"
        qo = q[:, :, rows]
        ko = kc[:, :, :Lk]
        vo = np.zeros((B, Hkv, Lk, D))
        vo[:, :, np.arange(Lk), np.arange(Lk)] = 1.0  # value j = e_j, so O = P
        r = oracle.causal(qo, ko, vo, scale=scale, bottom_right=not last)
        P = r["o"][..., :Lk]  # [B, Hq, M, Lk]
        for g in range(Hkv):
            out[:, g][:, rows, :Lk] = P[:, g * G : (g + 1) * G].sum(axis=1)
    return out


@pytest.mark.parametrize("Hq,Hkv,T,bs", [(2, 1, 40, 4), (6, 2, 37, 8), (4, 4, 33, 16), (8, 1, 64, 4)])
def test_scores_match_causal_attention_over_compressed_keys(Hq, Hkv, T, bs):
    B, D = 2, 16
    q = _rand((B, Hq, T, D), 3)
    kc = oracle.compress_mean(_rand((B, Hkv, T, D), 4), bs)
    scale = 0.37
    got = oracle.block_scores(q, kc, bs, scale=scale)
    want = _scores_via_causal_attention(q.numpy(), kc, bs, scale)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_scores_closed_forms_and_invariants():
    B, Hq, Hkv, T, D, bs = 1, 6, 2, 48, 8, 8
    G = Hq // Hkv
    q = _rand((B, Hq, T, D), 5)
    kc = oracle.compress_mean(_rand((B, Hkv, T, D), 6), bs)
    sc = oracle.block_scores(q, kc, bs)
    scale = 1.0 / math.sqrt(D)
    for t in range(T):
        nc = (t + 1) // bs
        if nc == 0:
            assert np.all(sc[:, :, t] == 0.0)  # no complete block yet
            continue
        np.testing.assert_allclose(sc[:, :, t, :nc].sum(-1), G, atol=1e-12)  # G probabilities
        assert np.all(sc[:, :, t, nc:] == 0.0)
        if nc == 1:  # one complete block: every head gives it probability 1
            np.testing.assert_allclose(sc[:, :, t, 0], G, atol=1e-12)
    # two complete blocks, G = 1: a sigmoid of the logit difference
    q1 = q[:, :1]
    sc1 = oracle.block_scores(q1, kc[:, :1], bs)
    t = 2 * bs - 1
    x = scale * float(q1[0, 0, t] @ torch.from_numpy(kc[0, 0, 0] - kc[0, 0, 1]))
    assert abs(sc1[0, 0, t, 0] - 1.0 / (1.0 + math.exp(-x))) < 1e-12
    # a shift common to every compressed key moves every logit of a row equally
    w = _rand((D,), 7).numpy()
    sc_shift = oracle.block_scores(q, kc + w, bs)
    np.testing.assert_allclose(sc_shift, sc, atol=1e-12)


def _topk_bruteforce(scores, bs, S, lens=None):
    """idx rows by Python's sort of the complete blocks by (-score, j)."""
    def key(x):
        return -math.inf if math.isnan(x) else x

    def row(sc, t):
        own, nc = t // bs, (t + 1) // bs
        cand = sorted((j for j in range(nc) if j != own), key=lambda j: (-key(float(sc[j])), j))
        r = [own] + cand[: S - 1]
        return r + [-1] * (S - len(r))

    if lens is None:
        B, Hkv, T, nb = scores.shape
        idx = np.full((B, Hkv, T, S), -1, dtype=np.int32)
        for b in range(B):
            for g in range(Hkv):
                for t in range(T):
                    idx[b, g, t] = row(scores[b, g, t], t)
        return idx
    total, Hkv, nb = scores.shape
    idx = np.full((total, Hkv, S), -1, dtype=np.int32)
    start = 0
    for L in lens:
        for t in range(L):
            for g in range(Hkv):
                idx[start + t, g] = row(scores[start + t, g], t)
        start += L
    return idx


@pytest.mark.parametrize("S", [1, 3, 6, 20])
def test_select_topk_matches_sorting(S):
    B, Hkv, T, bs = 2, 3, 45, 4
    nb = (T + bs - 1) // bs
    g = torch.Generator().manual_seed(8)
    # few distinct values so that ties are common, and some NaNs
    sc = torch.randint(0, 5, (B, Hkv, T, nb), generator=g).float() / 4
    sc[torch.rand(sc.shape, generator=g) < 0.05] = float("nan")
    sc = sc.numpy().astype(np.float32)
    got = oracle.select_topk(sc, bs, S)
    np.testing.assert_array_equal(got, _topk_bruteforce(sc, bs, S))
    assert oracle.validate_index(torch.from_numpy(got), bs) == 0


def test_select_topk_packed_sequences():
    bs, Hkv, S = 8, 2, 4
    lens = [20, 7, 33]
    total = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    nb = (max(lens) + bs - 1) // bs
    sc = _rand((total, Hkv, nb), 9).float().numpy()
    got = oracle.select_topk(sc, bs, S, cu_seqlens=cu)
    np.testing.assert_array_equal(got, _topk_bruteforce(sc, bs, S, lens))
    assert oracle.validate_index(torch.from_numpy(got), bs, cu_seqlens=torch.from_numpy(cu)) == 0


def test_select_topk_limits():
    B, Hkv, T, bs = 1, 1, 32, 4
    nb = T // bs
    sc = _rand((B, Hkv, T, nb), 10).numpy()
    one = oracle.select_topk(sc, bs, 1)
    np.testing.assert_array_equal(one[0, 0, :, 0], np.arange(T) // bs)  # own block only
    many = oracle.select_topk(sc, bs, nb + 2)
    for t in range(T):
        r = many[0, 0, t]
        nc, own = (t + 1) // bs, t // bs
        others = [j for j in range(nc) if j != own]
        assert r[0] == own
        assert sorted(r[1 : 1 + len(others)]) == others  # every complete block, once
        assert np.all(r[1 + len(others) :] == -1)
        vals = sc[0, 0, t, r[1 : 1 + len(others)]]
        assert np.all(np.diff(vals) <= 0)  # decreasing score


def test_selection_pipeline_gives_a_valid_index():
    B, Hq, Hkv, T, D, bs, S = 1, 4, 2, 50, 8, 8, 3
    q = _rand((B, Hq, T, D), 11)
    k = _rand((B, Hkv, T, D), 12)
    idx = oracle.select_topk(oracle.block_scores(q, oracle.compress_mean(k, bs), bs), bs, S)
    assert idx.shape == (B, Hkv, T, S)
    assert oracle.validate_index(torch.from_numpy(idx), bs) == 0
    o, lse = oracle.sel_fwd(q, k, k, torch.from_numpy(idx), bs)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


def test_planted_mistake_in_scores_is_caught():
    """Scores summed over the wrong heads (head h counted in kv group h % Hkv
    instead of h // G) must fail the pin against causal attention."""
    B, Hq, Hkv, T, D, bs = 1, 4, 2, 40, 16, 4
    q = _rand((B, Hq, T, D), 13)
    kc = oracle.compress_mean(_rand((B, Hkv, T, D), 14), bs)
    want = _scores_via_causal_attention(q.numpy(), kc, bs, 0.5)
    perm = [h for r in range(Hkv) for h in range(r, Hq, Hkv)]  # plant: h -> group h % Hkv
    bad = oracle.block_scores(q[:, perm], kc, bs, scale=0.5)
    assert np.max(np.abs(bad - want)) > 1e-3
