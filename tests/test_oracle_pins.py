"""Pins for the fp64 CPU oracle, against things other than itself.

Each pin targets a mistake the oracle could plausibly make:

* masked dense attention through torch's scaled_dot_product_attention +
  autograd (a library routine; selection attention is by definition dense
  attention under the mask "k <= t and k // bs in sel(t)", and the mask here
  is built by brute force from the index) -- catches wrong key sets, wrong
  GQA mapping, transposed operands, sign or scale errors in any gradient;
* central finite differences of L = <dO, O> -- the backward is the derivative
  of the forward;
* the dense causal special case against SDPA(is_causal=True);
* invariants fixed by the mathematics (sum_k dS = 0, sum dV = sum dO,
  sum dK = 0 per group);
* closed forms for rows with one attended key;
* -1 padding wherever it sits, slot order, empty rows;
* the inverse index against a pure-Python brute force;
* index validation cases;
* the sliding window (cuDNN-frontend page: the SDPA backward's window option)
  against SDPA with a brute-force band mask, its two limits (W >= T is plain
  causal attention, W = 1 attends the row's own key only), pair counts and
  sampled entries.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from block_sparse_attention_do_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore")


def _mask_from_idx(idx, T, bs):
    """bool [B, Hkv, T, T] mask by brute force over the index rows."""
    idx = idx.numpy()
    B, Hkv = idx.shape[:2]
    m = np.zeros((B, Hkv, T, T), dtype=bool)
    for b in range(B):
        for g in range(Hkv):
            for t in range(T):
                blocks = {int(j) for j in idx[b, g, t] if j >= 0}
                for k in range(t + 1):
                    if k // bs in blocks:
                        m[b, g, t, k] = True
    return torch.from_numpy(m)


def _sdpa_reference(q, k, v, do, mask_kv, scale):
    """fp64 masked attention + autograd via torch SDPA; mask per kv head."""
    G = q.shape[1] // k.shape[1]
    qr, kr, vr = (x.double().clone().requires_grad_(True) for x in (q, k, v))
    ke = kr.repeat_interleave(G, dim=1)
    ve = vr.repeat_interleave(G, dim=1)
    mask = mask_kv.repeat_interleave(G, dim=1)
    o = F.scaled_dot_product_attention(qr, ke, ve, attn_mask=mask, scale=scale)
    o.backward(do.double())
    return o.detach(), qr.grad, kr.grad, vr.grad


CASES = [
    # B, Hq, Hkv, T, D, bs, S
    (1, 2, 1, 32, 8, 4, 3),     # G=2
    (2, 3, 3, 29, 16, 8, 2),    # G=1, ragged tail (29 % 8)
    (1, 6, 2, 40, 8, 8, 8),     # G=3, S > valid blocks for every row
    (2, 4, 1, 33, 4, 16, 2),    # G=4, large block, ragged
]


@pytest.mark.parametrize("case", CASES)
def test_matches_masked_sdpa(case):
    B, Hq, Hkv, T, D, bs, S = case
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=7)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=3)
    scale = 1.0 / math.sqrt(D)
    mask = _mask_from_idx(idx, T, bs)
    o_ref, dq_ref, dk_ref, dv_ref = _sdpa_reference(q, k, v, do, mask, scale)
    o, lse = oracle.sel_fwd(q, k, v, idx, bs)
    r = oracle.sel_bwd(q, k, v, idx, do, bs)
    np.testing.assert_allclose(o, o_ref.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["o"], o_ref.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dq"], dq_ref.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(r["dk"], dk_ref.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(r["dv"], dv_ref.numpy(), rtol=0, atol=1e-11)
    # LSE: torch.logsumexp over the masked scores (library reduction)
    G = Hq // Hkv
    s = torch.einsum("bhtd,bhkd->bhtk", q.double(), k.double().repeat_interleave(G, 1)) * scale
    s = s.masked_fill(~mask.repeat_interleave(G, 1), -math.inf)
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


def test_finite_differences():
    """Central differences of L = <dO, O(q,k,v)> on every input coordinate."""
    B, Hq, Hkv, T, D, bs, S = 1, 4, 2, 12, 4, 4, 2
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=11)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=5)
    idx[0, 1, 9, 1] = -1  # a padded row
    q, k, v, do = (x.double().numpy() for x in (q, k, v, do))
    r = oracle.sel_bwd(q, k, v, idx, do, bs)
    h = 1e-6

    def loss(qq, kk, vv):
        o, _ = oracle.sel_fwd(qq, kk, vv, idx, bs)
        return float(np.sum(o * do))

    for name, x, g in (("q", q, r["dq"]), ("k", k, r["dk"]), ("v", v, r["dv"])):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[i] += h
            xm[i] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            fd[i] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(g, fd, rtol=0, atol=2e-8, err_msg=name)


@pytest.mark.parametrize("G", [1, 4])
def test_dense_selection_is_causal_sdpa(G):
    B, Hkv, T, D, bs = 2, 2, 37, 8, 8
    Hq = Hkv * G
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=2)
    idx = inputs.make_dense_block_idx(B, Hkv, T, bs)
    qr, kr, vr = (x.double().clone().requires_grad_(True) for x in (q, k, v))
    o = F.scaled_dot_product_attention(qr, kr.repeat_interleave(G, 1), vr.repeat_interleave(G, 1),
                                       is_causal=True)
    o.backward(do.double())
    r = oracle.sel_bwd(q, k, v, idx, do, bs)
    np.testing.assert_allclose(r["o"], o.detach().numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(r["dq"], qr.grad.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(r["dk"], kr.grad.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(r["dv"], vr.grad.numpy(), atol=1e-11, rtol=0)


def test_invariants():
    B, Hq, Hkv, T, D, bs, S = 2, 6, 2, 96, 16, 8, 4
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=4)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=4)
    r = oracle.sel_bwd(q, k, v, idx, do, bs, want_dsum=True)
    G = Hq // Hkv
    assert np.max(np.abs(r["dsum"])) < 1e-12
    dO = do.double().numpy()
    for b in range(B):
        for g in range(Hkv):
            sum_dv = r["dv"][b, g].sum(axis=0)
            sum_do = dO[b, g * G:(g + 1) * G].sum(axis=(0, 1))
            np.testing.assert_allclose(sum_dv, sum_do, atol=1e-10, rtol=0)
            assert np.max(np.abs(r["dk"][b, g].sum(axis=0))) < 1e-10
    # O is a convex combination of the attended values
    vmax = v.double().numpy().max()
    vmin = v.double().numpy().min()
    assert r["o"].max() <= vmax + 1e-12 and r["o"].min() >= vmin - 1e-12


def test_single_key_rows_closed_form():
    """S = 1 and t at a block start: the row attends only key t."""
    B, Hq, Hkv, T, D, bs, S = 1, 2, 1, 16, 8, 4, 1
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=9)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S)
    r = oracle.sel_bwd(q, k, v, idx, do, bs)
    qd, kd, vd = (x.double().numpy() for x in (q, k, v))
    scale = 1 / math.sqrt(D)
    for h in range(Hq):
        for t in range(0, T, bs):
            np.testing.assert_allclose(r["o"][0, h, t], vd[0, 0, t], atol=1e-14, rtol=0)
            assert abs(r["lse"][0, h, t] - scale * qd[0, h, t] @ kd[0, 0, t]) < 1e-13
            assert np.max(np.abs(r["dq"][0, h, t])) < 1e-14


def test_two_key_row_closed_form():
    """Row t = 1 attending keys {0, 1}: softmax of two scores is a sigmoid."""
    B, Hq, Hkv, T, D, bs, S = 1, 1, 1, 2, 4, 2, 1
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=1)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S)
    o, lse = oracle.sel_fwd(q, k, v, idx, bs)
    qd, kd, vd = (x.double().numpy()[0, 0] for x in (q, k, v))
    scale = 0.5
    s0, s1 = scale * qd[1] @ kd[0], scale * qd[1] @ kd[1]
    p1 = 1.0 / (1.0 + math.exp(s0 - s1))
    np.testing.assert_allclose(o[0, 0, 1], (1 - p1) * vd[0] + p1 * vd[1], atol=1e-14, rtol=0)
    assert abs(lse[0, 0, 1] - (s1 + math.log1p(math.exp(s0 - s1)))) < 1e-13


def test_padding_position_and_slot_order_do_not_matter():
    B, Hq, Hkv, T, D, bs, S = 1, 4, 2, 48, 8, 4, 4
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=6)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=6)
    base = oracle.sel_bwd(q, k, v, idx, do, bs)
    rng = np.random.default_rng(0)
    wide = np.full((B, Hkv, T, S + 3), -1, dtype=np.int32)
    for b in range(B):
        for g in range(Hkv):
            for t in range(T):
                perm = rng.permutation(S + 3)
                wide[b, g, t, perm[:S]] = idx[b, g, t].numpy()
    r = oracle.sel_bwd(q, k, v, torch.from_numpy(wide), do, bs)
    for key in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_allclose(r[key], base[key], atol=1e-13, rtol=0, err_msg=key)


def test_empty_row_contributes_nothing():
    B, Hq, Hkv, T, D, bs, S = 1, 2, 1, 24, 8, 4, 3
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=8)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=8)
    t0 = 13
    idx_empty = idx.clone()
    idx_empty[0, 0, t0] = -1
    r = oracle.sel_bwd(q, k, v, idx_empty, do, bs)
    assert np.all(r["o"][0, :, t0] == 0) and np.all(np.isneginf(r["lse"][0, :, t0]))
    assert np.all(r["dq"][0, :, t0] == 0)
    do_zero = do.clone()
    do_zero[0, :, t0] = 0
    ref = oracle.sel_bwd(q, k, v, idx, do_zero, bs)
    np.testing.assert_allclose(r["dk"], ref["dk"], atol=1e-13, rtol=0)
    np.testing.assert_allclose(r["dv"], ref["dv"], atol=1e-13, rtol=0)


def test_varlen_matches_per_sequence_sdpa():
    lengths = [7, 33, 20]
    Hq, Hkv, D, bs, S = 4, 2, 8, 8, 3
    total = sum(lengths)
    cu = inputs.cu_seqlens_from_lengths(lengths)
    q, k, v, do = inputs.make_qkv_do(1, Hq, Hkv, total, D, seed=12, layout="thd")
    idx = inputs.make_varlen_block_idx(lengths, Hkv, bs, S, seed=12)
    r = oracle.sel_bwd(q, k, v, idx, do, bs, cu_seqlens=cu)
    scale = 1 / math.sqrt(D)
    for i, L in enumerate(lengths):
        a, b_ = int(cu[i]), int(cu[i + 1])
        to_bhtd = lambda x: x[a:b_].permute(1, 0, 2).unsqueeze(0)  # noqa: E731
        idx_s = idx[a:b_].permute(1, 0, 2).unsqueeze(0)
        mask = _mask_from_idx(idx_s, L, bs)
        o_ref, dq_ref, dk_ref, dv_ref = _sdpa_reference(
            to_bhtd(q), to_bhtd(k), to_bhtd(v), to_bhtd(do), mask, scale)
        back = lambda x: x[0].permute(1, 0, 2).numpy()  # noqa: E731
        np.testing.assert_allclose(r["o"][a:b_], back(o_ref), atol=1e-12, rtol=0)
        np.testing.assert_allclose(r["dq"][a:b_], back(dq_ref), atol=1e-11, rtol=0)
        np.testing.assert_allclose(r["dk"][a:b_], back(dk_ref), atol=1e-11, rtol=0)
        np.testing.assert_allclose(r["dv"][a:b_], back(dv_ref), atol=1e-11, rtol=0)


def _csr_brute(idx_np, lengths, bs, nbmax):
    offsets, rows = [], []
    B = len(lengths)
    Hkv = idx_np[0].shape[1]
    for b in range(B):
        for g in range(Hkv):
            for j in range(nbmax):
                offsets.append(len(rows))
                for t in range(lengths[b]):
                    if j in set(idx_np[b][t, g].tolist()):
                        rows.append(t)
    offsets.append(len(rows))
    return np.array(offsets, dtype=np.int32), np.array(rows, dtype=np.int32)


def test_inverse_index_bruteforce_fixed_and_varlen():
    B, Hkv, T, bs, S = 2, 3, 50, 8, 4
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=13)
    off, rows, nbmax = oracle.inverse_index(idx, bs)
    per_b = [idx[b].permute(1, 0, 2).numpy() for b in range(B)]
    ref_off, ref_rows = _csr_brute(per_b, [T] * B, bs, nbmax)
    assert np.array_equal(off, ref_off) and np.array_equal(rows, ref_rows)
    assert off[-1] == int((idx >= 0).sum())

    lengths = [9, 40, 1, 17]
    cu = inputs.cu_seqlens_from_lengths(lengths)
    vidx = inputs.make_varlen_block_idx(lengths, Hkv, bs, S, seed=2)
    off, rows, nbmax = oracle.inverse_index(vidx, bs, cu_seqlens=cu)
    per_b = [vidx[int(cu[i]):int(cu[i + 1])].numpy() for i in range(len(lengths))]
    ref_off, ref_rows = _csr_brute(per_b, lengths, bs, nbmax)
    assert np.array_equal(off, ref_off) and np.array_equal(rows, ref_rows)


def test_validate_index_cases():
    B, Hkv, T, bs, S = 1, 1, 16, 4, 3
    idx = inputs.make_block_idx(B, Hkv, T, bs, S)
    assert oracle.validate_index(idx, bs) == 0
    bad = idx.clone()
    bad[0, 0, 5, 1] = 2          # future block for t=5 (own block is 1)
    assert oracle.validate_index(bad, bs) == 3
    bad = idx.clone()
    bad[0, 0, 9, 2] = bad[0, 0, 9, 0]  # duplicate
    assert oracle.validate_index(bad, bs) == 3
    bad = idx.clone()
    bad[0, 0, 3, 2] = -2
    assert oracle.validate_index(bad, bs) == 3
    ok = idx.clone()
    ok[0, 0, 12] = torch.tensor([-1, 0, -1], dtype=torch.int32)  # own block omitted: allowed
    assert oracle.validate_index(ok, bs) == 0


def test_count_pairs_matches_mask():
    B, Hq, Hkv, T, bs, S = 2, 6, 2, 45, 8, 3
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=1)
    mask = _mask_from_idx(idx, T, bs)
    assert oracle.count_pairs(idx, Hq, bs) == int(mask.sum()) * (Hq // Hkv)


def test_do_dot_and_sampled_entries_agree_with_whole_problem():
    B, Hq, Hkv, T, D, bs, S = 1, 4, 2, 40, 8, 8, 3
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=21)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=21)
    r = oracle.sel_bwd(q, k, v, idx, do, bs)
    dd = oracle.do_dot(r["o"], do)
    np.testing.assert_allclose(dd, np.einsum("bhtd,bhtd->bht", r["o"], do.double().numpy()),
                               atol=1e-13, rtol=0)
    rows = [(0, 1, 0), (0, 3, 39), (0, 2, 17)]
    o, lse, dq = oracle.sel_rows(q, k, v, idx, do, bs, rows)
    for i, (b, h, t) in enumerate(rows):
        np.testing.assert_allclose(o[i], r["o"][b, h, t], atol=1e-14, rtol=0)
        np.testing.assert_allclose(dq[i], r["dq"][b, h, t], atol=1e-14, rtol=0)
        assert abs(lse[i] - r["lse"][b, h, t]) < 1e-14
    keys = [(0, 0, 0), (0, 1, 39), (0, 1, 8)]
    dk, dv = oracle.sel_keys(q, k, v, idx, do, bs, keys)
    for i, (b, g, kk) in enumerate(keys):
        np.testing.assert_allclose(dk[i], r["dk"][b, g, kk], atol=1e-13, rtol=0)
        np.testing.assert_allclose(dv[i], r["dv"][b, g, kk], atol=1e-13, rtol=0)


def test_planted_mistake_is_caught(monkeypatch):
    """A transposed GQA mapping (h % Hkv instead of h // G) must fail the SDPA pin."""
    B, Hq, Hkv, T, D, bs, S = 1, 4, 2, 24, 8, 4, 2
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=3)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=3)
    mask = _mask_from_idx(idx, T, bs)
    o_ref, *_ = _sdpa_reference(q, k, v, do, mask, 1 / math.sqrt(D))
    # plant: permute heads so head h reads kv head h % Hkv
    perm = [h for r in range(Hkv) for h in range(r, Hq, Hkv)]
    o_bad, _ = oracle.sel_fwd(q[:, perm], k, v, idx, bs)
    inv = np.argsort(perm)
    assert np.max(np.abs(o_bad[:, inv] - o_ref.numpy())) > 1e-3


def _band_mask(B, Hkv, T, W):
    """bool [B, Hkv, T, T]: k <= t and t - k < W, by brute force."""
    m = np.zeros((B, Hkv, T, T), dtype=bool)
    for t in range(T):
        for k in range(T):
            if k <= t and t - k < W:
                m[:, :, t, k] = True
    return torch.from_numpy(m)


@pytest.mark.parametrize("W,G", [(5, 1), (13, 2), (8, 3), (1, 2)])
def test_window_matches_band_masked_sdpa(W, G):
    """Dense causal attention limited to the W most recent keys."""
    B, Hkv, T, D, bs = 2, 2, 37, 8, 8
    Hq = Hkv * G
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=4)
    idx = inputs.make_dense_block_idx(B, Hkv, T, bs)
    scale = 1 / math.sqrt(D)
    o_ref, dq_ref, dk_ref, dv_ref = _sdpa_reference(q, k, v, do, _band_mask(B, Hkv, T, W), scale)
    r = oracle.sel_bwd(q, k, v, idx, do, bs, window=W)
    np.testing.assert_allclose(r["o"], o_ref.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(r["dq"], dq_ref.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(r["dk"], dk_ref.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(r["dv"], dv_ref.numpy(), atol=1e-11, rtol=0)
    o, lse = oracle.sel_fwd(q, k, v, idx, bs, window=W)
    np.testing.assert_allclose(o, o_ref.numpy(), atol=1e-12, rtol=0)
    assert oracle.count_pairs(idx, Hq, bs, window=W) == int(_band_mask(B, Hkv, T, W).sum()) * G


def test_window_limits():
    B, Hq, Hkv, T, D, bs = 1, 4, 2, 30, 8, 4
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=6)
    idx = inputs.make_dense_block_idx(B, Hkv, T, bs)
    full = oracle.sel_bwd(q, k, v, idx, do, bs)
    wide = oracle.sel_bwd(q, k, v, idx, do, bs, window=T)
    for n in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_array_equal(wide[n], full[n])
    # W = 1: each row sees its own key: O_t = v_t, LSE_t = scale q_t.k_t,
    # P = 1 so dS = 0: no dQ / dK; dV_k = sum over the group's heads of dO_k
    one = oracle.sel_bwd(q, k, v, idx, do, bs, window=1)
    G = Hq // Hkv
    vv = v.double().repeat_interleave(G, 1).numpy()
    np.testing.assert_allclose(one["o"], vv, atol=1e-14, rtol=0)
    sc = (q.double() * k.double().repeat_interleave(G, 1)).sum(-1).numpy() / math.sqrt(D)
    np.testing.assert_allclose(one["lse"], sc, atol=1e-13, rtol=0)
    np.testing.assert_allclose(one["dq"], 0.0, atol=1e-14)
    np.testing.assert_allclose(one["dk"], 0.0, atol=1e-14)
    dv_ref = do.double().reshape(B, Hkv, G, T, D).sum(2).numpy()
    np.testing.assert_allclose(one["dv"], dv_ref, atol=1e-13, rtol=0)


def test_window_sampled_entries_agree_with_whole_problem():
    B, Hq, Hkv, T, D, bs, W = 1, 4, 2, 41, 8, 8, 11
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=8)
    idx = inputs.make_dense_block_idx(B, Hkv, T, bs)
    r = oracle.sel_bwd(q, k, v, idx, do, bs, window=W)
    rows = [(0, 0, 0), (0, 3, 10), (0, 1, 11), (0, 2, 40)]
    o, lse, dq = oracle.sel_rows(q, k, v, idx, do, bs, rows, window=W)
    for i, (b, h, t) in enumerate(rows):
        np.testing.assert_allclose(o[i], r["o"][b, h, t], atol=1e-13, rtol=0)
        np.testing.assert_allclose(dq[i], r["dq"][b, h, t], atol=1e-13, rtol=0)
    keys = [(0, 0, 0), (0, 1, 29), (0, 0, 30), (0, 1, 40)]
    dk, dv = oracle.sel_keys(q, k, v, idx, do, bs, keys, window=W)
    for i, (b, g, kk) in enumerate(keys):
        np.testing.assert_allclose(dk[i], r["dk"][b, g, kk], atol=1e-13, rtol=0)
        np.testing.assert_allclose(dv[i], r["dv"][b, g, kk], atol=1e-13, rtol=0)


# ---- attention sinks: one logit per query head in every row's denominator


def _sink_reference(q, k, v, do, mask_kv, sinks, scale):
    """fp64 attention with a sink column appended to the scores, by plain
    torch ops + autograd (softmax over [scores | sink], the sink's
    probability dropped before P.V)."""
    G = q.shape[1] // k.shape[1]
    qr, kr, vr = (x.double().clone().requires_grad_(True) for x in (q, k, v))
    sr = torch.as_tensor(sinks, dtype=torch.float64).clone().requires_grad_(True)
    ke = kr.repeat_interleave(G, dim=1)
    ve = vr.repeat_interleave(G, dim=1)
    mask = mask_kv.repeat_interleave(G, dim=1)
    s = torch.einsum("bhtd,bhkd->bhtk", qr, ke) * scale
    s = s.masked_fill(~mask, float("-inf"))
    B, Hq, T, _ = s.shape
    col = sr.view(1, Hq, 1, 1).expand(B, Hq, T, 1)
    p = torch.softmax(torch.cat([s, col], dim=-1), dim=-1)[..., :T]
    o = torch.einsum("bhtk,bhkd->bhtd", p, ve)
    lse = torch.logsumexp(torch.cat([s, col], dim=-1), dim=-1)
    o.backward(do.double())
    return o.detach(), lse.detach(), qr.grad, kr.grad, vr.grad, sr.grad


@pytest.mark.parametrize("W,G", [(0, 2), (7, 1), (0, 3)])
def test_sinks_match_autograd(W, G):
    """Dense causal (optionally windowed) attention with sinks against plain
    torch fp64 attention with an appended sink column and its autograd."""
    B, Hkv, T, D, bs = 2, 2, 29, 8, 4
    Hq = Hkv * G
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=8)
    idx = inputs.make_dense_block_idx(B, Hkv, T, bs)
    sinks = np.random.default_rng(3).normal(0.0, 2.0, Hq)
    scale = 1 / math.sqrt(D)
    mask = _band_mask(B, Hkv, T, W if W else T + 1)
    o_ref, lse_ref, dq_ref, dk_ref, dv_ref, ds_ref = _sink_reference(q, k, v, do, mask, sinks, scale)
    r = oracle.sel_bwd(q, k, v, idx, do, bs, window=W, sinks=sinks)
    np.testing.assert_allclose(r["o"], o_ref.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(r["lse"], lse_ref.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(r["dq"], dq_ref.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(r["dk"], dk_ref.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(r["dv"], dv_ref.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(r["dsinks"], ds_ref.numpy(), atol=1e-10, rtol=0)
    o, lse = oracle.sel_fwd(q, k, v, idx, bs, window=W, sinks=sinks)
    np.testing.assert_array_equal(o, r["o"])
    np.testing.assert_array_equal(lse, r["lse"])


def test_sinks_closed_forms_and_finite_differences():
    B, Hq, Hkv, T, D, bs = 1, 2, 1, 12, 4, 4
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=10)
    idx = inputs.make_dense_block_idx(B, Hkv, T, bs)
    sinks = np.array([0.7, -1.3])
    scale = 1 / math.sqrt(D)
    r = oracle.sel_bwd(q, k, v, idx, do, bs, sinks=sinks)
    # row t = 0 sees key 0 only: LSE = log(e^s + e^sigma), O = v_0 / (1 + e^(sigma - s))
    qd, kd, vd = (x.double().numpy() for x in (q, k, v))
    for h in range(Hq):
        s00 = scale * float(qd[0, h, 0] @ kd[0, 0, 0])
        assert abs(r["lse"][0, h, 0] - np.logaddexp(s00, sinks[h])) < 1e-13
        np.testing.assert_allclose(r["o"][0, h, 0], vd[0, 0, 0] / (1 + math.exp(sinks[h] - s00)), atol=1e-13)
    # sigma -> -inf: no sink at all
    none = oracle.sel_bwd(q, k, v, idx, do, bs)
    far = oracle.sel_bwd(q, k, v, idx, do, bs, sinks=np.full(Hq, -np.inf))
    for n in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_array_equal(far[n], none[n])
    np.testing.assert_array_equal(far["dsinks"], np.zeros(Hq))
    # central differences of <dO, O(sigma)>
    dod = do.double().numpy()
    eps = 1e-6
    for h in range(Hq):
        sp, sm = sinks.copy(), sinks.copy()
        sp[h] += eps
        sm[h] -= eps
        fp = float((oracle.sel_fwd(q, k, v, idx, bs, sinks=sp)[0] * dod).sum())
        fm = float((oracle.sel_fwd(q, k, v, idx, bs, sinks=sm)[0] * dod).sum())
        assert abs((fp - fm) / (2 * eps) - r["dsinks"][h]) < 1e-7


# ---- whole-block sampling (oracle.sel_blocks), used where the full-size
# workloads are too large for the whole-output oracle


def test_sampled_blocks_against_masked_sdpa():
    """dK/dV of whole blocks, against masked SDPA + autograd: the first block
    (selected by nearly every row), a middle block, a ragged last block and a
    block whose keys no row reaches (an empty list gives zeros)."""
    B, Hq, Hkv, T, D, bs, S = 2, 6, 2, 45, 8, 8, 3
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=23)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=23)
    idx[1, 0, :, :] = torch.where(idx[1, 0] == 2, torch.full_like(idx[1, 0], -1), idx[1, 0])  # nobody keeps block 2
    mask = _mask_from_idx(idx, T, bs)
    _, _, dk_ref, dv_ref = _sdpa_reference(q, k, v, do, mask, 1.0 / math.sqrt(D))
    blocks = [(0, 0, 0), (0, 1, 3), (1, 1, 5), (1, 0, 2), (0, 1, 5)]
    dk, dv = oracle.sel_blocks(q, k, v, idx, do, bs, blocks)
    for i, (b, g, j) in enumerate(blocks):
        n = min(bs, T - j * bs)
        np.testing.assert_allclose(dk[i, :n], dk_ref[b, g, j * bs:j * bs + n].numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv[i, :n], dv_ref[b, g, j * bs:j * bs + n].numpy(), rtol=0, atol=1e-12)
        assert not np.any(dk[i, n:]) and not np.any(dv[i, n:])
    assert not np.any(dk[3]) and not np.any(dv[3])


def test_sampled_blocks_varlen_and_window():
    """The packed layout (per-sequence SDPA) and the sliding window (band
    mask), block by block."""
    lengths = [19, 5, 30]
    Hq, Hkv, D, bs, S = 4, 2, 8, 8, 3
    cu = inputs.cu_seqlens_from_lengths(lengths)
    q, k, v, do = inputs.make_qkv_do(1, Hq, Hkv, sum(lengths), D, seed=24, layout="thd")
    idx = inputs.make_varlen_block_idx(lengths, Hkv, bs, S, seed=24)
    blocks = [(0, 0, 0), (0, 1, 2), (1, 0, 0), (2, 1, 1), (2, 0, 3)]
    dk, dv = oracle.sel_blocks(q, k, v, idx, do, bs, blocks, cu_seqlens=cu)
    for i, (b, g, j) in enumerate(blocks):
        a, L = int(cu[b]), lengths[b]
        sub = lambda x: x[a:a + L].permute(1, 0, 2).unsqueeze(0)  # [1, H, L, D]
        m = _mask_from_idx(idx[a:a + L].permute(1, 0, 2).unsqueeze(0), L, bs)
        _, _, dk_ref, dv_ref = _sdpa_reference(sub(q), sub(k), sub(v), sub(do), m, 1.0 / math.sqrt(D))
        n = min(bs, L - j * bs)
        np.testing.assert_allclose(dk[i, :n], dk_ref[0, g, j * bs:j * bs + n].numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv[i, :n], dv_ref[0, g, j * bs:j * bs + n].numpy(), rtol=0, atol=1e-12)
    # window 11 on the dense index, fixed length
    B, T, W = 1, 41, 11
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=25)
    idx = inputs.make_dense_block_idx(B, Hkv, T, bs)
    band = torch.zeros(B, Hkv, T, T, dtype=torch.bool)
    for t in range(T):
        band[:, :, t, max(0, t - W + 1):t + 1] = True
    _, _, dk_ref, dv_ref = _sdpa_reference(q, k, v, do, band, 1.0 / math.sqrt(D))
    blocks = [(0, 0, 0), (0, 1, 2), (0, 0, 5)]
    dk, dv = oracle.sel_blocks(q, k, v, idx, do, bs, blocks, window=W)
    for i, (b, g, j) in enumerate(blocks):
        n = min(bs, T - j * bs)
        np.testing.assert_allclose(dk[i, :n], dk_ref[b, g, j * bs:j * bs + n].numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv[i, :n], dv_ref[b, g, j * bs:j * bs + n].numpy(), rtol=0, atol=1e-12)


# ---- dense causal attention with separate query and key lengths (top-left
# and bottom-right alignment of the diagonal, optional window): oracle.causal


def _sdpa_bias(q, k, v, do, mask):
    """fp64 SDPA + autograd, GQA by repeating kv heads; mask [Tq, Tk] bool or
    a torch attention-bias object."""
    G = q.shape[1] // k.shape[1]
    qr, kr, vr = (x.double().clone().requires_grad_(True) for x in (q, k, v))
    o = F.scaled_dot_product_attention(qr, kr.repeat_interleave(G, 1), vr.repeat_interleave(G, 1), attn_mask=mask)
    o.backward(do.double())
    return o.detach(), qr.grad, kr.grad, vr.grad


@pytest.mark.parametrize("Tq,Tk", [(5, 12), (12, 12), (9, 30)])
def test_causal_bottom_right_matches_torch_lower_right_bias(Tq, Tk):
    """Bottom-right alignment (Lk >= Lq: every row attends something) against
    torch's own lower-right causal bias, forward and gradients."""
    from torch.nn.attention.bias import causal_lower_right

    B, Hq, Hkv, D = 2, 4, 2, 8
    q, _, _, do = inputs.make_qkv_do(B, Hq, Hkv, Tq, D, seed=40)
    _, k, v, _ = inputs.make_qkv_do(B, Hq, Hkv, Tk, D, seed=41)
    r = oracle.causal(q, k, v, do, bottom_right=True)
    o, dq, dk, dv = _sdpa_bias(q, k, v, do, causal_lower_right(Tq, Tk))
    for name, ref in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        np.testing.assert_allclose(r[name], ref.numpy(), rtol=0, atol=1e-12, err_msg=name)


@pytest.mark.parametrize("Tq,Tk", [(5, 12), (12, 7)])
def test_causal_top_left_matches_sdpa_is_causal(Tq, Tk):
    """Top-left alignment with unequal lengths: SDPA's is_causal (the
    upper-left diagonal)."""
    B, Hq, Hkv, D = 1, 4, 1, 8
    q, _, _, do = inputs.make_qkv_do(B, Hq, Hkv, Tq, D, seed=42)
    _, k, v, _ = inputs.make_qkv_do(B, Hq, Hkv, Tk, D, seed=43)
    r = oracle.causal(q, k, v, do, bottom_right=False)
    G = Hq // Hkv
    qr, kr, vr = (x.double().clone().requires_grad_(True) for x in (q, k, v))
    o = F.scaled_dot_product_attention(qr, kr.repeat_interleave(G, 1), vr.repeat_interleave(G, 1), is_causal=True)
    o.backward(do.double())
    for name, ref in (("o", o.detach()), ("dq", qr.grad), ("dk", kr.grad), ("dv", vr.grad)):
        np.testing.assert_allclose(r[name], ref.numpy(), rtol=0, atol=1e-12, err_msg=name)


def test_causal_bottom_right_empty_rows_and_window():
    """Lq > Lk, bottom-right: the first Lq - Lk rows attend nothing (O = 0,
    LSE = -inf, no gradient); the others match SDPA on a brute-force mask
    c_t = t + Lk - Lq, with a window of 3 keys."""
    B, Hq, Hkv, D, Tq, Tk, W = 1, 2, 1, 8, 10, 6, 3
    q, _, _, do = inputs.make_qkv_do(B, Hq, Hkv, Tq, D, seed=44)
    _, k, v, _ = inputs.make_qkv_do(B, Hq, Hkv, Tk, D, seed=45)
    r = oracle.causal(q, k, v, do, bottom_right=True, window=W)
    shift = Tk - Tq
    mask = torch.zeros(Tq, Tk, dtype=torch.bool)
    for t in range(Tq):
        for kk in range(Tk):
            c = t + shift
            mask[t, kk] = kk <= c and c - kk < W
    live = mask.any(1)
    assert not live[: Tq - Tk].any() and live[Tq - Tk:].all()
    assert np.all(r["o"][:, :, ~live.numpy()] == 0) and np.all(np.isneginf(r["lse"][:, :, ~live.numpy()]))
    assert np.all(r["dq"][:, :, ~live.numpy()] == 0)
    ql, dol = q[:, :, live], do[:, :, live]
    o, dq, dk, dv = _sdpa_bias(ql, k, v, dol, mask[live])
    np.testing.assert_allclose(r["o"][:, :, live.numpy()], o.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dq"][:, :, live.numpy()], dq.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dk"], dk.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dv"], dv.numpy(), rtol=0, atol=1e-12)


def test_causal_packed_sequences_and_equal_length_reduction():
    """Packed sequences with their own Lq, Lk against the fixed-length oracle
    per sequence; and with Lq = Lk both alignments reduce to the selection
    oracle's dense case."""
    lq, lk = [3, 7, 5], [8, 7, 2]
    Hq, Hkv, D = 4, 2, 8
    cuq, cuk = inputs.cu_seqlens_from_lengths(lq), inputs.cu_seqlens_from_lengths(lk)
    q, _, _, do = inputs.make_qkv_do(1, Hq, Hkv, sum(lq), D, seed=46, layout="thd")
    _, k, v, _ = inputs.make_qkv_do(1, Hq, Hkv, sum(lk), D, seed=47, layout="thd")
    for br in (False, True):
        r = oracle.causal(q, k, v, do, cu_seqlens_q=cuq, cu_seqlens_k=cuk, bottom_right=br)
        for b in range(3):
            a, e, ka, ke = int(cuq[b]), int(cuq[b + 1]), int(cuk[b]), int(cuk[b + 1])
            sub = lambda x: x.permute(1, 0, 2).unsqueeze(0)
            rb = oracle.causal(sub(q[a:e]), sub(k[ka:ke]), sub(v[ka:ke]), sub(do[a:e]), bottom_right=br)
            np.testing.assert_allclose(r["o"][a:e], rb["o"][0].transpose(1, 0, 2), rtol=0, atol=1e-14)
            np.testing.assert_allclose(r["dk"][ka:ke], rb["dk"][0].transpose(1, 0, 2), rtol=0, atol=1e-14)
    B, T, bs = 2, 21, 4
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, seed=48)
    ref = oracle.sel_bwd(q, k, v, inputs.make_dense_block_idx(B, Hkv, T, bs), do, bs, window=5)
    for br in (False, True):
        r = oracle.causal(q, k, v, do, bottom_right=br, window=5)
        for name in ("o", "dq", "dk", "dv"):
            np.testing.assert_allclose(r[name], ref[name], rtol=0, atol=1e-13, err_msg=name)
