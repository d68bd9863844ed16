"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Inputs are seeded and synthetic (block_sparse_attention_do_gb300.inputs); the
oracle reads the same dtype-rounded values.  The gate is the gradcheck page's
TOL table applied as a max-abs bound (tests/golden/gate_tolerances.json):
2e-3 for fp32, 6e-2 for bf16 beyond the rounding of a bf16 output (see
_maxerr); the inverse index must match bit-exactly.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_do_gb300 import api, inputs

pytestmark = pytest.mark.gpu

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "gate_tolerances.json")))
TOL = {torch.float32: GOLD["max_abs_gate"]["fp32"], torch.bfloat16: GOLD["max_abs_gate"]["bf16"]}
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_sparse_attention_do_gb300 import build

    build.build()
    api.lib()


def _rawerr(got, ref):
    """Plain max-abs error."""
    if not ref.size:
        return 0.0
    return float(np.max(np.abs(got.double().cpu().numpy() - ref)))


def _maxerr(got, ref):
    """Max-abs error beyond the rounding of the stored output.

    A bf16 output carries its own round-to-nearest error, up to half an ulp:
    bf16 has an 8-bit significand, so its unit roundoff is 2^-8 and the
    rounding error of x is at most 2^-8 |x|.  We allow 2^-8 * |ref| per
    element for it, so the atol gate bounds the computation's error.  This
    matters only where gradients are far from unit scale (dK/dV summed over
    many heads, G >= 64); the gate's page states its tolerance for unit-scale
    gradients.  fp32 outputs get no allowance.
    """
    if not ref.size:
        return 0.0
    g = got.double().cpu().numpy()
    err = np.abs(g - ref)
    if got.dtype == torch.bfloat16:
        err = err - 2.0 ** -8 * np.abs(ref)
    return float(np.max(err))


def _log_errors(label, errs, raw):
    """Appends the case's errors to the file NSA_PARITY_LOG names (if set):
    the record of which cases pass the plain max-abs gate and which need the
    bf16 output-rounding allowance."""
    path = os.environ.get("NSA_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": label, "gated": errs, "raw": raw}) + "\n")


def _run(q, k, v, do, idx, bs, cu=None, dense=False, window=None):
    g = [x.to(DEV) for x in (q, k, v, do)]
    gi = None if (dense or window is not None) else idx.to(DEV)
    gcu = None if cu is None else cu.to(DEV)
    o, lse = api.sel_fwd(g[0], g[1], g[2], gi, bs, cu_seqlens=gcu, dense=dense, window=window)
    dq, dk, dv = api.sel_bwd(g[0], g[1], g[2], o, g[3], lse, gi, bs, cu_seqlens=gcu, dense=dense,
                             window=window)
    torch.cuda.synchronize()
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)


def _compare(got, ref, dtype, names=("o", "dq", "dk", "dv"), label=None):
    tol = TOL[dtype]
    errs = {n: _maxerr(got[n], ref[n]) for n in names}
    raw = {n: _rawerr(got[n], ref[n]) for n in names}
    lse_ref = ref["lse"]
    lse_got = got["lse"].double().cpu().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lse_got)), "empty rows must give -inf"
    errs["lse"] = raw["lse"] = float(np.max(np.abs(lse_got[fin] - lse_ref[fin]))) if fin.any() else 0.0
    _log_errors(label or os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], errs, raw)
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, f"max-abs errors over {tol}: {errs} (raw max-abs, no rounding allowance: {raw})"
    return errs


SMALL = [
    # B, Hq, Hkv, T, D, bs, S
    (1, 2, 1, 128, 32, 16, 4),    # the small fp32 fwd+bwd workload
    (1, 3, 3, 77, 64, 32, 3),     # G=1, ragged tail
    (2, 6, 2, 200, 64, 32, 8),    # G=3, S above the valid count for early rows
    (1, 4, 1, 150, 128, 64, 3),   # G=4, D=128, bs=64, ragged
    (1, 16, 1, 256, 128, 64, 4),  # G=16
    (1, 32, 1, 300, 128, 64, 5),  # G=32, ragged
    (2, 32, 2, 200, 128, 64, 3),  # G=16, two kv heads, batch 2
    (1, 16, 2, 333, 128, 64, 6),  # G=8: 16 tokens a tile
    (1, 48, 2, 260, 128, 64, 5),  # G=24: 5 tokens, 120 of 128 rows used
    (1, 64, 1, 130, 128, 64, 3),  # G=64: 2 tokens a tile
    (1, 128, 1, 70, 128, 64, 2),  # G=128: one token a tile
    (1, 4, 1, 1100, 64, 16, 40),  # S above 32: the per-slot index checks
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("case", SMALL)
def test_small_selection(case, dtype):
    B, Hq, Hkv, T, D, bs, S = case
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=dtype, seed=1)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=1)
    got = _run(q, k, v, do, idx, bs)
    ref = oracle.sel_bwd(q, k, v, idx, do, bs)
    _compare(got, ref, dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_padding_anywhere_and_empty_rows(dtype):
    B, Hq, Hkv, T, D, bs, S = 1, 4, 2, 192, 64, 32, 5
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=dtype, seed=5)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=5)
    rng = np.random.default_rng(0)
    a = idx.numpy()
    for g in range(Hkv):
        for t in range(T):
            a[0, g, t] = a[0, g, t][rng.permutation(S)]  # -1 anywhere, own block anywhere
    a[0, 0, 100] = -1      # an empty row
    a[0, 1, 37, :] = -1
    a[0, 1, 37, 2] = 0     # a row attending only an earlier block
    idx = torch.from_numpy(a)
    got = _run(q, k, v, do, idx, bs)
    ref = oracle.sel_bwd(q, k, v, idx, do, bs)
    _compare(got, ref, dtype)


def test_padding_and_empty_rows_tensor_core_shapes():
    """The bf16 tensor-core kernels (D=128, block 64, G=16) on -1 slots anywhere,
    rows with no selected block and rows holding only an earlier block."""
    B, Hq, Hkv, T, D, bs, S = 1, 32, 2, 320, 128, 64, 4
    dtype = torch.bfloat16
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=dtype, seed=15)
    a = inputs.make_block_idx(B, Hkv, T, bs, S, seed=15).numpy()
    rng = np.random.default_rng(1)
    for g in range(Hkv):
        for t in range(T):
            a[0, g, t] = a[0, g, t][rng.permutation(S)]
    a[0, 0, 200] = -1
    a[0, 1, 7] = -1
    a[0, 1, 300, :] = -1
    a[0, 1, 300, 3] = 2
    idx = torch.from_numpy(a)
    got = _run(q, k, v, do, idx, bs)
    ref = oracle.sel_bwd(q, k, v, idx, do, bs)
    _compare(got, ref, dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_dense_causal(dtype):
    B, Hq, Hkv, T, D, bs = 2, 8, 2, 200, 128, 64
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=dtype, seed=2)
    idx = inputs.make_dense_block_idx(B, Hkv, T, bs)
    got = _run(q, k, v, do, None, bs, dense=True)
    ref = oracle.sel_bwd(q, k, v, idx, do, bs)
    _compare(got, ref, dtype)


@pytest.mark.parametrize("dtype,Hq", [(torch.float32, 8), (torch.bfloat16, 8), (torch.bfloat16, 32)])
def test_varlen(dtype, Hq):
    lengths = [130, 1, 64, 257, 90]
    Hkv, D, bs, S = 2, 128, 64, 3
    total = sum(lengths)
    cu = inputs.cu_seqlens_from_lengths(lengths)
    q, k, v, do = inputs.make_qkv_do(1, Hq, Hkv, total, D, dtype=dtype, seed=3, layout="thd")
    idx = inputs.make_varlen_block_idx(lengths, Hkv, bs, S, seed=3)
    got = _run(q, k, v, do, idx, bs, cu=cu)
    ref = oracle.sel_bwd(q, k, v, idx, do, bs, cu_seqlens=cu)
    _compare(got, ref, dtype)


@pytest.mark.parametrize("dtype,shape,W", [
    (torch.bfloat16, (1, 16, 1, 300, 128, 64, 1), 100),  # tensor cores; the window edge cuts blocks
    (torch.bfloat16, (1, 16, 1, 300, 128, 64, 1), 64),   # window = one block
    (torch.bfloat16, (2, 32, 2, 200, 128, 64, 1), 1),    # own key only
    (torch.bfloat16, (1, 16, 1, 300, 128, 64, 1), 1000), # wider than T: dense causal
    (torch.float32, (2, 6, 2, 150, 64, 32, 1), 45),      # other shapes: split-precision tensor cores
    (torch.bfloat16, (1, 4, 1, 150, 128, 64, 1), 70),    # G = 4: head-major tiles, cp.async gathers
])
def test_sliding_window(dtype, shape, W):
    B, Hq, Hkv, T, D, bs, _ = shape
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=dtype, seed=14)
    idx = inputs.make_dense_block_idx(B, Hkv, T, bs)
    got = _run(q, k, v, do, None, bs, window=W)
    ref = oracle.sel_bwd(q, k, v, idx, do, bs, window=W)
    _compare(got, ref, dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_sliding_window_varlen(dtype):
    lengths = [130, 1, 64, 257, 90]
    Hq, Hkv, D, bs, W = 16, 1, 128, 64, 75
    total = sum(lengths)
    cu = inputs.cu_seqlens_from_lengths(lengths)
    q, k, v, do = inputs.make_qkv_do(1, Hq, Hkv, total, D, dtype=dtype, seed=15, layout="thd")
    nb = (max(lengths) + bs - 1) // bs
    # the oracle's dense index: every block up to the token's own
    dense = np.full((total, Hkv, nb), -1, dtype=np.int32)
    off = 0
    for L in lengths:
        for t in range(L):
            dense[off + t, :, : t // bs + 1] = np.arange(t // bs + 1)
        off += L
    got = _run(q, k, v, do, None, bs, cu=cu, window=W)
    ref = oracle.sel_bwd(q, k, v, torch.from_numpy(dense), do, bs, cu_seqlens=cu, window=W)
    _compare(got, ref, dtype)


def test_inverse_index_bit_exact():
    for (B, Hkv, T, bs, S, lengths) in ((2, 3, 333, 32, 6, None), (0, 2, 0, 64, 5, [70, 1, 300])):
        if lengths is None:
            idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=4)
            cu = None
        else:
            idx = inputs.make_varlen_block_idx(lengths, Hkv, bs, S, seed=4)
            cu = inputs.cu_seqlens_from_lengths(lengths)
        off, rows, ws = api.build_inverse_index(idx.to(DEV), Hkv * 2, bs,
                                                cu_seqlens=None if cu is None else cu.to(DEV))
        ref_off, ref_rows, _ = oracle.inverse_index(idx, bs, cu_seqlens=cu)
        off = off.cpu().numpy()
        assert np.array_equal(off, ref_off)
        assert np.array_equal(rows[: off[-1]].cpu().numpy(), ref_rows)
        assert api.get_error(ws) == 0


def test_do_dot():
    gen = torch.Generator().manual_seed(22)
    o = torch.randn(2, 3, 100, 128, generator=gen).to(torch.bfloat16)
    do = torch.randn(2, 3, 100, 128, generator=gen).to(torch.bfloat16)
    got = api.do_dot(o.to(DEV), do.to(DEV)).cpu().double().numpy()
    ref = oracle.do_dot(o, do)
    assert np.max(np.abs(got - ref)) < 1e-3


@pytest.mark.parametrize("S", [3, 40])
def test_bad_index_is_reported(S):
    B, Hq, Hkv, T, D, bs = 1, 2, 1, 128, 64, 32
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.bfloat16)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S)
    cases = []
    bad = idx.clone()
    bad[0, 0, 10, 1] = 3       # future block
    cases.append(bad)
    bad = idx.clone()
    bad[0, 0, 100, 2] = bad[0, 0, 100, 0]  # repeated block
    cases.append(bad)
    bad = idx.clone()
    bad[0, 0, 50, 1] = -7
    cases.append(bad)
    for bad in cases:
        assert oracle.validate_index(bad, bs) == 3
        g = [x.to(DEV) for x in (q, k, v, do, bad)]
        ws = torch.empty(api.bwd_workspace_size(api.problem_from(g[0], g[1], bs, S)),
                         dtype=torch.uint8, device=DEV)
        o, lse = api.sel_fwd(g[0], g[1], g[2], g[4], bs, ws=ws)
        assert api.get_error(ws) == 3
        api.sel_bwd(g[0], g[1], g[2], o, g[3], lse, g[4], bs, ws=ws)
        assert api.get_error(ws) == 3
        assert api.get_error(ws) == 0  # reading clears it


def test_runs_on_the_callers_stream():
    B, Hq, Hkv, T, D, bs, S = 1, 4, 1, 256, 128, 64, 4
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.bfloat16, seed=9)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=9)
    g = [x.to(DEV) for x in (q, k, v, do, idx)]
    ref = _run(q, k, v, do, idx, bs)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = api.sel_fwd(g[0], g[1], g[2], g[4], bs, stream=s)
        dq, dk, dv = api.sel_bwd(g[0], g[1], g[2], o, g[3], lse, g[4], bs, stream=s)
    s.synchronize()
    for name, x in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.equal(x, ref[name]), f"{name} differs between streams (must be deterministic)"


def test_other_shapes_ordered_on_the_callers_stream():
    """The other-shapes backward runs its dQ on a helper stream forked from
    the caller's: it must start after the caller's earlier work (dO written
    there behind a GPU wait) and end before the caller's later work (a copy
    of dq), and give the same bits as the same call on the default stream."""
    B, Hq, Hkv, T, D, bs, S = 2, 6, 2, 1024, 64, 32, 8
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.bfloat16, seed=61)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=61)
    ref = _run(q, k, v, do, idx, bs)
    g = [x.to(DEV) for x in (q, k, v, do, idx)]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    do_late = torch.zeros_like(g[3])
    with torch.cuda.stream(s):
        torch.cuda._sleep(20_000_000)  # ~10 ms of GPU time before dO exists
        do_late.copy_(g[3])
        dq, dk, dv = api.sel_bwd(g[0], g[1], g[2], ref["o"], do_late, ref["lse"], g[4], bs, stream=s)
        after = [x.clone() for x in (dq, dk, dv)]
    s.synchronize()
    for name, x in zip(("dq", "dk", "dv"), after):
        assert torch.equal(x, ref[name]), f"{name}: not ordered on the caller's stream"


@pytest.mark.parametrize("shape", [
    (1, 4, 1, 256, 128, 64, 4),   # tensor-core kernels for D = 128, 64-key blocks
    (2, 6, 2, 1024, 64, 32, 8),   # the other shapes (dQ on the helper stream)
])
def test_backward_captured_in_a_cuda_graph(shape):
    """Forward and backward captured once into a CUDA graph and replayed on
    new inputs give the same bits as direct calls."""
    B, Hq, Hkv, T, D, bs, S = shape
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.bfloat16, seed=62)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=62)
    q2, k2, v2, do2 = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.bfloat16, seed=63)
    ref = _run(q2, k2, v2, do2, idx, bs)
    bufs = [x.to(DEV) for x in (q, k, v, do)]
    gi = idx.to(DEV)

    def step():
        o, lse = api.sel_fwd(bufs[0], bufs[1], bufs[2], gi, bs)
        return (o, lse) + tuple(api.sel_bwd(bufs[0], bufs[1], bufs[2], o, bufs[3], lse, gi, bs))

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture (workspaces, kernel attributes)
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        outs = step()
    for dst, src in zip(bufs, (q2, k2, v2, do2)):
        dst.copy_(src.to(DEV))
    graph.replay()
    torch.cuda.synchronize()
    for name, x in zip(("o", "lse", "dq", "dk", "dv"), outs):
        assert torch.equal(x, ref[name]), f"{name} differs under graph replay"


def test_count_pairs():
    B, Hq, Hkv, T, bs, S = 2, 6, 2, 500, 32, 6
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=6)
    assert api.count_pairs(idx.to(DEV), Hq, bs) == oracle.count_pairs(idx, Hq, bs)


def test_deterministic_bitwise():
    B, Hq, Hkv, T, D, bs, S = 1, 16, 1, 512, 128, 64, 4
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.bfloat16, seed=10)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=10)
    a = _run(q, k, v, do, idx, bs)
    b = _run(q, k, v, do, idx, bs)
    for n in ("o", "lse", "dq", "dk", "dv"):
        assert torch.equal(a[n], b[n]), n


def test_outputs_only_16_byte_aligned():
    """o and dq at addresses 16- but not 32-byte aligned (all the API asks) take
    the kernels' 16-byte store path: bitwise the results of the 32-byte one."""
    import ctypes as C
    B, Hq, Hkv, T, D, bs, S = 1, 16, 1, 1100, 128, 64, 16
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.bfloat16, seed=12)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=12)
    q, k, v, do, idx = (x.cuda() for x in (q, k, v, do, idx))
    o_ref, lse_ref = api.sel_fwd(q, k, v, idx, bs)
    dq_ref, dk_ref, dv_ref = api.sel_bwd(q, k, v, o_ref, do, lse_ref, idx, bs)[:3]

    def shifted_like(x):  # 8 bf16 = 16 bytes past a 256-byte aligned allocation
        y = torch.empty(x.numel() + 8, dtype=x.dtype, device=x.device)[8:].view_as(x)
        assert y.data_ptr() % 32 == 16
        return y

    o2, lse2 = shifted_like(q), torch.empty_like(lse_ref)
    p = api.problem_from(q, k, bs, S)
    ws = torch.empty(api.fwd_workspace_size(p), dtype=torch.uint8, device="cuda")
    s = api.lib().nsa_sel_fwd(C.byref(p), api._ptr(q), api._ptr(k), api._ptr(v), api._ptr(idx), api._ptr(o2),
                              api._ptr(lse2), api._ptr(ws), ws.numel(), api._stream(None))
    assert s == 0
    torch.cuda.synchronize()
    assert api.get_error(ws) == 0
    assert torch.equal(o2, o_ref) and torch.equal(lse2, lse_ref)
    dq2 = shifted_like(q)
    api.sel_bwd(q, k, v, o_ref, do, lse_ref, idx, bs, out=(dq2, torch.empty_like(k), torch.empty_like(v)))
    torch.cuda.synchronize()
    assert torch.equal(dq2, dq_ref)


@pytest.mark.parametrize("dtype,shape", [
    (torch.bfloat16, (1, 16, 1, 1024, 128, 64, 4)),   # tensor-core path
    (torch.float32, (2, 6, 2, 300, 64, 32, 5)),       # SIMT path
])
def test_planned_backward_is_the_same_backward(dtype, shape):
    """A plan built once gives bitwise the results of the plain backward, and
    is only read: two calls on one plan agree."""
    B, Hq, Hkv, T, D, bs, S = shape
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=dtype, seed=12)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=12)
    ref = _run(q, k, v, do, idx, bs)
    g = [x.to(DEV) for x in (q, k, v, do, idx)]
    plan = api.build_plan(g[0], g[1], g[4], bs)
    assert api.get_error(plan) == 0
    want = oracle.sel_bwd(q, k, v, idx, do, bs)
    for _ in range(2):
        dq, dk, dv = api.sel_bwd(g[0], g[1], g[2], ref["o"], g[3], ref["lse"], g[4], bs, plan=plan)
        torch.cuda.synchronize()
        for name, x in (("dq", dq), ("dk", dk), ("dv", dv)):
            assert torch.equal(x, ref[name]), name
        # and the planned backward itself against the oracle
        _compare(dict(o=ref["o"], lse=ref["lse"], dq=dq, dk=dk, dv=dv), want, dtype)


def _clustered_block_idx(B, Hkv, T, bs, S, seed):
    """Each token: its own block, then up to S - 1 distinct earlier blocks
    drawn from a few shared sets (every token of a set of consecutive tokens
    draws from the same 6 blocks), -1 padding.  Tokens share most of their
    blocks, so tile grouping meets many equal costs."""
    g = np.random.default_rng(seed)
    idx = np.full((B, Hkv, T, S), -1, dtype=np.int32)
    for b in range(B):
        for h in range(Hkv):
            for t0 in range(0, T, 24):
                own0 = t0 // bs
                pool = g.choice(max(own0, 1), size=min(6, max(own0, 1)), replace=False) if own0 else np.array([], int)
                for t in range(t0, min(T, t0 + 24)):
                    own = t // bs
                    cand = [int(j) for j in pool if j < own]
                    picks = g.permutation(cand)[: S - 1] if cand else []
                    row = [own] + [int(j) for j in picks]
                    idx[b, h, t, : len(row)] = row
    return torch.from_numpy(idx)


def test_grouped_query_tiles_clustered_selection():
    """Clustered selections on the tensor-core path (G = 16, BHTD), where the
    forward, the backward and a plan group the query tiles by shared blocks:
    forward, backward and planned backward against the oracle."""
    B, Hq, Hkv, T, D, bs, S = 1, 32, 2, 700, 128, 64, 5
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.bfloat16, seed=70)
    idx = _clustered_block_idx(B, Hkv, T, bs, S, seed=70)
    assert oracle.validate_index(idx, bs) == 0
    got = _run(q, k, v, do, idx, bs)
    ref = oracle.sel_bwd(q, k, v, idx, do, bs)
    _compare(got, ref, torch.bfloat16)
    g = [x.to(DEV) for x in (q, k, v, do, idx)]
    plan = api.build_plan(g[0], g[1], g[4], bs)
    dq, dk, dv = api.sel_bwd(g[0], g[1], g[2], got["o"], g[3], got["lse"], g[4], bs, plan=plan)
    torch.cuda.synchronize()
    assert api.get_error(plan) == 0
    _compare(dict(o=got["o"], lse=got["lse"], dq=dq, dk=dk, dv=dv), ref, torch.bfloat16)


def test_planned_backward_varlen_and_bad_index():
    Hq, Hkv, D, bs, S = 8, 2, 128, 64, 6
    lengths = [130, 64, 257]
    cu = inputs.cu_seqlens_from_lengths(lengths)
    total = int(cu[-1])
    q, k, v, do = inputs.make_qkv_do(1, Hq, Hkv, total, D, dtype=torch.bfloat16, seed=13, layout="thd")
    idx = inputs.make_varlen_block_idx(lengths, Hkv, bs, S, seed=13)
    ref = _run(q, k, v, do, idx, bs, cu=cu)
    g = [x.to(DEV) for x in (q, k, v, do, idx)]
    gcu = cu.to(DEV)
    plan = api.build_plan(g[0], g[1], g[4], bs, cu_seqlens=gcu)
    dq, dk, dv = api.sel_bwd(g[0], g[1], g[2], ref["o"], g[3], ref["lse"], g[4], bs, cu_seqlens=gcu,
                             plan=plan)
    torch.cuda.synchronize()
    for name, x in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.equal(x, ref[name]), name
    want = oracle.sel_bwd(q, k, v, idx, do, bs, cu_seqlens=cu)
    _compare(dict(o=ref["o"], lse=ref["lse"], dq=dq, dk=dk, dv=dv), want, torch.bfloat16)
    bad = idx.clone()
    bad[5, 0, 1] = 3  # a future block of the first sequence
    plan = api.build_plan(g[0], g[1], bad.to(DEV), bs, cu_seqlens=gcu)
    assert api.get_error(plan) == 3


def test_realistic_sparsity_tensor_core_path():
    """16 blocks, 4 slots: tiles walk a block union much larger than each
    token's selection (the per-token bitmaps and warp skips matter)."""
    B, Hq, Hkv, T, D, bs, S = 1, 16, 1, 1024, 128, 64, 4
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.bfloat16, seed=17)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=17)
    got = _run(q, k, v, do, idx, bs)
    ref = oracle.sel_bwd(q, k, v, idx, do, bs)
    _compare(got, ref, torch.bfloat16)
    off, rows, ws = api.build_inverse_index(idx.to(DEV), Hq, bs)
    ref_off, ref_rows, _ = oracle.inverse_index(idx, bs)
    assert np.array_equal(off.cpu().numpy(), ref_off)
    assert np.array_equal(rows[: int(ref_off[-1])].cpu().numpy(), ref_rows)


def _unit_tokens(G):
    """Tokens per dK/dV work unit of the tensor-core path: 128 row tiles of
    128 // G tokens (one token for G >= 128).  A block whose token list is
    longer is split over several units whose fp32 partials a second kernel
    sums; the tests below make sure such blocks are compared whole."""
    return (1 if G >= 128 else 128 // G) * 128


def _list_lengths(idx, bs, cu=None):
    """[(b, g, j, number of tokens selecting block j)] from the oracle's
    inverse index."""
    off, _, nb = oracle.inverse_index(idx, bs, cu_seqlens=cu)
    Hkv = idx.shape[1]  # [B, Hkv, T, S] or packed [total, Hkv, S]
    n = np.diff(off.astype(np.int64))
    out = []
    for x, c in enumerate(n):
        bg, j = divmod(x, nb)
        out.append((bg // Hkv, bg % Hkv, j, int(c)))
    return out


def _sample_rows(rng, B, Hq, Hkv, lengths, n, tile_tokens):
    """n (b, h, t) rows: the sequence edges and block boundaries, then every
    (token, head) position of a 128-row query tile in turn (token tl of the
    tile, head hh of the group) at random tiles, sequences and kv heads."""
    G = Hq // Hkv
    rows = []
    for b in range(B):
        L = lengths[b]
        for t in (0, L - 1, 63, 64, L // 2):
            rows.append((b, int(rng.integers(0, Hq)), min(t, L - 1)))
    i = 0
    while len(rows) < n:
        pos = i % (tile_tokens * G)
        tl, hh = divmod(pos, G)
        b = int(rng.integers(0, B))
        L = lengths[b]
        ntiles = (L + tile_tokens - 1) // tile_tokens
        t = min(int(rng.integers(0, ntiles)) * tile_tokens + tl, L - 1)
        rows.append((b, int(rng.integers(0, Hkv)) * G + hh, t))
        i += 1
    return rows


def _sample_blocks(rng, lists, G, bs, lengths, n_split=4):
    """Whole kv blocks to compare: every sequence's last two blocks (few
    selecting rows), block 0 and the most selected block, and random blocks
    among those whose list is split over several dK/dV units."""
    unit = _unit_tokens(G)
    split = [(b, g, j) for b, g, j, c in lists if c > unit]
    by_len = sorted(lists, key=lambda x: -x[3])
    blocks = {(b, g, j) for b, g, j, _ in by_len[:1]}
    blocks.add((0, 0, 0))
    for x in rng.permutation(len(split))[:n_split]:
        blocks.add(split[int(x)])
    Hkv = max(g for _, g, _, _ in lists) + 1
    for b, L in enumerate(lengths[:2]):
        last = (L - 1) // bs
        blocks.add((b, int(rng.integers(0, Hkv)), last))
        if last > 0:
            blocks.add((b, 0, last - 1))
    return sorted(blocks), len(split)


def _full_size_check(q, k, v, do, idx, bs, cu=None, dense=False, n_rows=256, min_split=0):
    """Sampled outputs of a full-size run against the oracle: n_rows query
    rows (o, lse, dq) over every row position of a query tile, and whole kv
    blocks (dk, dv of all their keys) including blocks split over several
    dK/dV units; plus identities that hold over the whole output."""
    got = _run(q, k, v, do, idx, bs, cu=cu, dense=dense)
    tol = TOL[torch.bfloat16]
    thd = cu is not None
    if thd:
        lengths = [int(cu[i + 1] - cu[i]) for i in range(len(cu) - 1)]
        B, Hq = len(lengths), q.shape[1]
    else:
        B, Hq, T = q.shape[0], q.shape[1], q.shape[2]
        lengths = [T] * B
    Hkv = k.shape[1]
    G = Hq // Hkv
    rng = np.random.default_rng(0)
    Tq = 1 if G >= 128 else 128 // G
    rows = _sample_rows(rng, B, Hq, Hkv, lengths, n_rows, Tq)
    o, lse, dq = oracle.sel_rows(q, k, v, idx, do, bs, rows, cu_seqlens=cu)

    def at(x, b, h, t):
        return x[int(cu[b]) + t, h] if thd else x[b, h, t]

    worst = {"o": 0.0, "dq": 0.0, "lse": 0.0, "dk": 0.0, "dv": 0.0}
    for i, (b, h, t) in enumerate(rows):
        eo = float(np.max(np.abs(at(got["o"], b, h, t).double().cpu().numpy() - o[i])))
        eq = float(np.max(np.abs(at(got["dq"], b, h, t).double().cpu().numpy() - dq[i])))
        el = abs(float(at(got["lse"], b, h, t)) - lse[i])
        worst["o"], worst["dq"], worst["lse"] = max(worst["o"], eo), max(worst["dq"], eq), max(worst["lse"], el)
        assert eo <= tol and eq <= tol and el <= tol, ((b, h, t), eo, eq, el)
    # whole blocks, split ones included
    lists = _list_lengths(idx, bs, cu)
    blocks, n_split = _sample_blocks(rng, lists, G, bs, lengths)
    assert n_split >= min_split, f"expected at least {min_split} split blocks, found {n_split}"
    dk, dv = oracle.sel_blocks(q, k, v, idx, do, bs, blocks, cu_seqlens=cu)
    for i, (b, g, j) in enumerate(blocks):
        nk = min(bs, lengths[b] - j * bs)
        for name, ref in (("dk", dk[i, :nk]), ("dv", dv[i, :nk])):
            x = got[name]
            blk = (x[int(cu[b]) + j * bs:int(cu[b]) + j * bs + nk, g] if thd else x[b, g, j * bs:j * bs + nk])
            e = float(np.max(np.abs(blk.double().cpu().numpy() - ref)))
            worst[name] = max(worst[name], e)
            assert e <= tol, (name, (b, g, j), e)
    _log_errors(os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0],
                {"sampled_rows": len(rows), "blocks": len(blocks), "split_blocks_in_problem": n_split}, worst)
    # identities over every output: sum_keys dV = sum of the group's dO over
    # rows that attend anything; sum_keys dK = 0 (rows of P sum to 1 and
    # rows of dS sum to 0).  Each dK/dV entry carries its bf16 rounding (at
    # most 2^-8 of itself), so a sum may be off by up to 2^-8 sum_k |entry|;
    # never less than 0.5 is allowed.
    dvs, dks, dos = got["dv"].double().cpu(), got["dk"].double().cpu(), do.double()
    fin = torch.isfinite(got["lse"].cpu())

    def check(dv_keys, dk_keys, want):
        tv = torch.clamp(2.0 ** -8 * dv_keys.abs().sum(0), min=0.5)
        tk = torch.clamp(2.0 ** -8 * dk_keys.abs().sum(0), min=0.5)
        assert torch.all(torch.abs(dv_keys.sum(0) - want) <= tv)
        assert torch.all(torch.abs(dk_keys.sum(0)) <= tk)

    if thd:
        for b in range(B):
            a, e = int(cu[b]), int(cu[b + 1])
            for g in range(Hkv):
                sel = fin[a:e, g * G:(g + 1) * G].unsqueeze(-1)
                check(dvs[a:e, g], dks[a:e, g], (dos[a:e, g * G:(g + 1) * G] * sel).sum(dim=(0, 1)))
    else:
        for b in range(B):
            for g in range(Hkv):
                sel = fin[b, g * G:(g + 1) * G].unsqueeze(-1)
                check(dvs[b, g], dks[b, g], (dos[b, g * G:(g + 1) * G] * sel).sum(dim=(0, 1)))


@pytest.mark.parametrize("shape", [
    (1, 32, 1, 1100, 128, 64, 16),  # G=32: 512-token units; blocks 0-15 split in three
    (1, 128, 1, 400, 128, 64, 4),   # G=128: 128-token units
    (1, 16, 1, 1100, 128, 64, 16),  # G=16: 1024-token units; block 0 splits in two
])
def test_split_blocks_whole_output(shape):
    """Blocks selected by more tokens than one dK/dV unit holds: their units
    write fp32 partials that the reduction kernel adds.  Whole outputs
    against the oracle."""
    B, Hq, Hkv, T, D, bs, S = shape
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.bfloat16, seed=19)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=19)
    unit = _unit_tokens(Hq // Hkv)
    lists = _list_lengths(idx, bs)
    assert sum(c > unit for *_, c in lists) >= 1, "the shape must split a block"
    got = _run(q, k, v, do, idx, bs)
    ref = oracle.sel_bwd(q, k, v, idx, do, bs)
    _compare(got, ref, torch.bfloat16)


def test_split_blocks_planned_backward():
    """The same split blocks through a plan built once (nsa_plan_build):
    against the oracle."""
    B, Hq, Hkv, T, D, bs, S = 1, 32, 1, 1100, 128, 64, 16
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.bfloat16, seed=20)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=20)
    g = [x.to(DEV) for x in (q, k, v, do, idx)]
    o, lse = api.sel_fwd(g[0], g[1], g[2], g[4], bs)
    plan = api.build_plan(g[0], g[1], g[4], bs)
    dq, dk, dv = api.sel_bwd(g[0], g[1], g[2], o, g[3], lse, g[4], bs, plan=plan)
    torch.cuda.synchronize()
    assert api.get_error(plan) == 0
    ref = oracle.sel_bwd(q, k, v, idx, do, bs)
    _compare(dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv), ref, torch.bfloat16)


def test_full_size_long_sequence_sampled():
    """B=1 Hq=32 Hkv=2 T=8192 D=128 block 64 S=16, bf16 (the benchmark workload)."""
    B, Hq, Hkv, T, D, bs, S = 1, 32, 2, 8192, 128, 64, 16
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.bfloat16, seed=0)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=0)
    _full_size_check(q, k, v, do, idx, bs, min_split=50)


def test_full_size_very_long_sequence_sampled():
    """B=1 Hq=16 Hkv=1 T=65536 D=128 block 64 S=16, bf16: 1024 selectable
    blocks per row, so the query-tile kernels' union buffers no longer fit
    twice beside three K stages (the fewer-stage / single-buffer layouts)."""
    B, Hq, Hkv, T, D, bs, S = 1, 16, 1, 65536, 128, 64, 16
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.bfloat16, seed=3)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=3)
    _full_size_check(q, k, v, do, idx, bs, min_split=50)


def test_full_size_dense_causal_sampled():
    """B=2 Hq=32 Hkv=8 T=4096 D=128 block 64, every valid block selected."""
    B, Hq, Hkv, T, D, bs = 2, 32, 8, 4096, 128, 64
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.bfloat16, seed=0)
    idx = inputs.make_dense_block_idx(B, Hkv, T, bs)
    _full_size_check(q, k, v, do, idx, bs, dense=True)


def test_full_size_varlen_sampled():
    """8 packed sequences with lengths uniform in [128, 4096], Hq=32 Hkv=8
    D=128 block 64 S=16."""
    lengths = inputs.make_varlen_lengths(8, 128, 4096, seed=0)
    Hq, Hkv, D, bs, S = 32, 8, 128, 64, 16
    cu = inputs.cu_seqlens_from_lengths(lengths)
    q, k, v, do = inputs.make_qkv_do(1, Hq, Hkv, sum(lengths), D, dtype=torch.bfloat16, seed=0,
                                     layout="thd")
    idx = inputs.make_varlen_block_idx(lengths, Hkv, bs, S, seed=0)
    _full_size_check(q, k, v, do, idx, bs, cu=cu)


def test_full_size_mid_size_fp32_and_bf16():
    """B=2 Hq=6 Hkv=2 (G=3) T=1024 D=64 block 32 S=8 in fp32 and bf16, whole
    outputs against the oracle."""
    B, Hq, Hkv, T, D, bs, S = 2, 6, 2, 1024, 64, 32, 8
    for dtype in (torch.float32, torch.bfloat16):
        q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=dtype, seed=0)
        idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=0)
        got = _run(q, k, v, do, idx, bs)
        ref = oracle.sel_bwd(q, k, v, idx, do, bs)
        _compare(got, ref, dtype)


# ---- attention sinks on the dense entry (tensor-core path for bf16 D=128
# bs=64, SIMT otherwise), against the oracle with the same sinks

SINK_CASES = [
    # dtype, (B, Hq, Hkv, T, D, bs), window, thd
    (torch.bfloat16, (1, 16, 1, 300, 128, 64), 0, False),
    (torch.bfloat16, (2, 8, 2, 200, 128, 64), 96, False),
    (torch.float32, (1, 4, 2, 150, 64, 32), 0, False),
    (torch.bfloat16, (0, 16, 2, 0, 128, 64), 0, True),  # THD, lengths below
]


@pytest.mark.parametrize("dtype,shape,window,thd", SINK_CASES)
def test_sinks_dense(dtype, shape, window, thd):
    B, Hq, Hkv, T, D, bs = shape
    sinks = torch.from_numpy(np.random.default_rng(11).normal(0.0, 2.0, Hq).astype(np.float32))
    if thd:
        lens = [130, 1, 257, 64]
        cu = inputs.cu_seqlens_from_lengths(lens)
        total = sum(lens)
        q, k, v, do = inputs.make_qkv_do(1, Hq, Hkv, total, D, dtype=dtype, seed=12, layout="thd")
        nb = (max(lens) + bs - 1) // bs
        dense = np.full((total, Hkv, nb), -1, dtype=np.int32)  # every block up to the token's own
        off = 0
        for L in lens:
            for t in range(L):
                dense[off + t, :, : t // bs + 1] = np.arange(t // bs + 1)
            off += L
        ref = oracle.sel_bwd(q, k, v, torch.from_numpy(dense), do, bs, cu_seqlens=cu, window=window,
                             sinks=sinks.numpy())
        gcu = cu.to(DEV)
    else:
        q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=dtype, seed=12)
        ref = oracle.sel_bwd(q, k, v, inputs.make_dense_block_idx(B, Hkv, T, bs), do, bs, window=window,
                             sinks=sinks.numpy())
        gcu = None
    g = [x.to(DEV) for x in (q, k, v, do)]
    gs = sinks.to(DEV)
    o, lse = api.sel_fwd(g[0], g[1], g[2], None, bs, cu_seqlens=gcu, window=window or None, sinks=gs)
    dq, dk, dv, dsinks = api.sel_bwd(g[0], g[1], g[2], o, g[3], lse, None, bs, cu_seqlens=gcu,
                                     window=window or None, sinks=gs)
    torch.cuda.synchronize()
    _compare(dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv), ref, dtype)
    got = dsinks.cpu().double().numpy()
    tol = TOL[dtype]
    assert np.all(np.abs(got - ref["dsinks"]) <= tol * np.maximum(1.0, np.abs(ref["dsinks"]))), \
        (got, ref["dsinks"])


# ---- declared strides: q, k, v (and dq, dk, dv) as views of packed tensors


def _packed_views(x_q, x_k, x_v, thd, pad_tokens=0):
    """q, k, v copied into one packed tensor ([B, T(+pad), Hq + 2 Hkv, D], or
    [total, Hq + 2 Hkv, D]) and returned as non-contiguous views of it."""
    if thd:
        total, Hq, D = x_q.shape
        Hkv = x_k.shape[1]
        pk = torch.empty(total, Hq + 2 * Hkv, D, dtype=x_q.dtype, device=DEV)
        q, k, v = pk[:, :Hq], pk[:, Hq:Hq + Hkv], pk[:, Hq + Hkv:]
    else:
        B, Hq, T, D = x_q.shape
        Hkv = x_k.shape[1]
        pk = torch.zeros(B, T + pad_tokens, Hq + 2 * Hkv, D, dtype=x_q.dtype, device=DEV)
        q = pk[:, :T, :Hq].transpose(1, 2)
        k = pk[:, :T, Hq:Hq + Hkv].transpose(1, 2)
        v = pk[:, :T, Hq + Hkv:].transpose(1, 2)
    q.copy_(x_q)
    k.copy_(x_k)
    v.copy_(x_v)
    assert not q.is_contiguous() and not k.is_contiguous()
    return q, k, v


@pytest.mark.parametrize("dtype,shape,pad", [
    (torch.bfloat16, (2, 32, 2, 300, 128, 64, 4), 0),  # tensor cores, row-gather maps (batch folded into tokens)
    (torch.bfloat16, (2, 8, 2, 200, 128, 64, 3), 0),   # tensor cores, G = 4: tile maps and cp.async gathers
    (torch.float32, (2, 6, 2, 150, 64, 32, 3), 0),     # other shapes: split-precision tensor cores
    (torch.bfloat16, (2, 16, 1, 130, 128, 64, 3), 8),  # padded token capacity: batch folds nowhere (other shapes)
])
def test_declared_strides_packed_qkv(dtype, shape, pad):
    """q, k, v are views of one packed [B, T, Hq + 2 Hkv, D] tensor and
    dq, dk, dv views of another: the kernels read and write them in place
    through the declared strides, and the results match the oracle."""
    B, Hq, Hkv, T, D, bs, S = shape
    xq, xk, xv, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=dtype, seed=26)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=26)
    q, k, v = _packed_views(xq.to(DEV), xk.to(DEV), xv.to(DEV), False, pad)
    dq, dk, dv = _packed_views(torch.zeros_like(xq, device=DEV), torch.zeros_like(xk, device=DEV),
                               torch.zeros_like(xv, device=DEV), False, pad)
    gi, gdo = idx.to(DEV), do.to(DEV)
    o, lse = api.sel_fwd(q, k, v, gi, bs)
    api.sel_bwd(q, k, v, o, gdo, lse, gi, bs, out=(dq, dk, dv))
    torch.cuda.synchronize()
    ref = oracle.sel_bwd(xq, xk, xv, idx, do, bs)
    _compare(dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv), ref, dtype)


def test_declared_strides_packed_thd():
    """The packed variable-length layout with q, k, v (and the gradients) as
    views of one [total, Hq + 2 Hkv, D] tensor; o and dO as views too."""
    lengths = [130, 1, 64, 257, 90]
    Hq, Hkv, D, bs, S = 32, 2, 128, 64, 4
    cu = inputs.cu_seqlens_from_lengths(lengths)
    total = sum(lengths)
    xq, xk, xv, do = inputs.make_qkv_do(1, Hq, Hkv, total, D, dtype=torch.bfloat16, seed=27, layout="thd")
    idx = inputs.make_varlen_block_idx(lengths, Hkv, bs, S, seed=27)
    q, k, v = _packed_views(xq.to(DEV), xk.to(DEV), xv.to(DEV), True)
    dq, dk, dv = _packed_views(torch.zeros_like(xq, device=DEV), torch.zeros_like(xk, device=DEV),
                               torch.zeros_like(xv, device=DEV), True)
    # o and dO interleaved in one [total, 2 Hq, D] tensor
    od = torch.empty(total, 2 * Hq, D, dtype=torch.bfloat16, device=DEV)
    o_view, do_view = od[:, :Hq], od[:, Hq:]
    do_view.copy_(do.to(DEV))
    gi, gcu = idx.to(DEV), cu.to(DEV)
    o, lse = api.sel_fwd(q, k, v, gi, bs, cu_seqlens=gcu)
    o_view.copy_(o)
    api.sel_bwd(q, k, v, o_view, do_view, lse, gi, bs, cu_seqlens=gcu, out=(dq, dk, dv))
    torch.cuda.synchronize()
    ref = oracle.sel_bwd(xq, xk, xv, idx, do, bs, cu_seqlens=cu)
    _compare(dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv), ref, torch.bfloat16)


# ---- dense causal attention with keys of their own lengths (nsa_causal_*):
# top-left and bottom-right alignment of the diagonal, with a window


CAUSAL_CASES = [
    # dtype, (B, Hq, Hkv, D, bs), q lengths, k lengths (None: BHTD with Tq, Tk), bottom_right, window
    (torch.bfloat16, (2, 16, 1, 128, 64), 200, 333, True, 0),     # tensor cores, G = 16, Lk > Lq
    (torch.bfloat16, (1, 32, 2, 128, 64), 300, 130, True, 0),     # Lq > Lk: the first 170 rows see nothing
    (torch.bfloat16, (1, 16, 2, 128, 64), 150, 260, False, 0),    # top-left: keys past Lq unused
    (torch.bfloat16, (1, 8, 2, 128, 64), 300, 500, True, 100),    # G = 4 (cp.async gathers), window
    (torch.float32, (2, 6, 2, 64, 32), 100, 150, True, 40),       # other shapes, split precision
    (torch.bfloat16, (0, 8, 2, 128, 64), [130, 1, 64, 257], [200, 64, 1, 257], True, 70),   # THD
    (torch.bfloat16, (0, 32, 2, 128, 64), [300, 90], [40, 300], True, 0),                   # THD, G = 16
    (torch.float32, (0, 4, 2, 64, 32), [50, 7], [80, 3], False, 0),                          # THD, other shapes
]


@pytest.mark.parametrize("dtype,shape,lq,lk,br,window", CAUSAL_CASES)
def test_causal_own_key_lengths(dtype, shape, lq, lk, br, window):
    B, Hq, Hkv, D, bs = shape
    if isinstance(lq, list):
        cuq, cuk = inputs.cu_seqlens_from_lengths(lq), inputs.cu_seqlens_from_lengths(lk)
        q, _, _, do = inputs.make_qkv_do(1, Hq, Hkv, sum(lq), D, dtype=dtype, seed=50, layout="thd")
        _, k, v, _ = inputs.make_qkv_do(1, Hq, Hkv, sum(lk), D, dtype=dtype, seed=51, layout="thd")
        gcq, gck = cuq.to(DEV), cuk.to(DEV)
    else:
        cuq = cuk = gcq = gck = None
        q, _, _, do = inputs.make_qkv_do(B, Hq, Hkv, lq, D, dtype=dtype, seed=50)
        _, k, v, _ = inputs.make_qkv_do(B, Hq, Hkv, lk, D, dtype=dtype, seed=51)
    g = [x.to(DEV) for x in (q, k, v, do)]
    kw = dict(block_size=bs, window=window, bottom_right=br, cu_seqlens_q=gcq, cu_seqlens_k=gck)
    o, lse = api.causal_fwd(g[0], g[1], g[2], **kw)
    dq, dk, dv = api.causal_bwd(g[0], g[1], g[2], o, g[3], lse, **kw)
    torch.cuda.synchronize()
    ref = oracle.causal(q, k, v, do, cu_seqlens_q=cuq, cu_seqlens_k=cuk, window=window, bottom_right=br)
    _compare(dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv), ref, dtype)


# ---- the other shapes on tensor cores (k_gtc.cu): D 32/64/128 x blocks of
# 16/32/64 in bf16, D 32/64 in fp32 by split precision


@pytest.mark.parametrize("dtype,shape", [
    (torch.float32, (2, 6, 2, 1024, 64, 32, 8)),    # the mid-size workload in fp32 (split precision)
    (torch.bfloat16, (2, 6, 2, 1024, 64, 32, 8)),   # ... and in bf16
    (torch.float32, (1, 2, 1, 128, 32, 16, 4)),     # the small fp32 fwd+bwd workload
    (torch.bfloat16, (1, 16, 2, 300, 128, 32, 6)),  # D = 128, 32-key blocks
    (torch.bfloat16, (2, 8, 1, 257, 32, 64, 3)),    # D = 32 (padded), 64-key blocks, G = 8
    # 175 query tiles of 8 tokens, more than the GPU has SMs: the launches that
    # keep two CTAs per SM (forward in both types, dQ in bf16)
    (torch.bfloat16, (1, 16, 1, 1400, 64, 32, 6)),
    (torch.float32, (1, 16, 1, 1400, 64, 32, 6)),
])
def test_other_shapes_run_on_tensor_cores(dtype, shape):
    """These shapes launch the tensor-core kernels of k_gtc.cu (seen through
    the library's per-launch tracer), not the CUDA-core ones, and match the
    oracle."""
    B, Hq, Hkv, T, D, bs, S = shape
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=dtype, seed=60)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=60)
    api.trace_enable(64)
    api.trace_reset()
    try:
        got = _run(q, k, v, do, idx, bs)
        names = {n for n, _ in api.trace_records()}
    finally:
        api.trace_enable(0)
    assert {"fwd_gtc", "dkdv_gtc", "dq_gtc"} <= names, names
    assert not any(n.endswith("_simt") for n in names), names
    ref = oracle.sel_bwd(q, k, v, idx, do, bs)
    _compare(got, ref, dtype)
