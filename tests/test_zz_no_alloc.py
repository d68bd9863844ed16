"""nsa_build_inverse_index_noalloc: the inverse-index builder for callers that
cannot allocate device memory when they call the library (their memory is
fixed at start-up, or an allocation would stall their stream schedule).  It
keeps its scratch in a fixed array inside the library instead of a caller
workspace.

Its results must equal those of nsa_build_inverse_index (integer output, so
bit for bit), on two calls in a row: the second call meets the array still
holding the first call's contents.  This file sorts last so that a failing
run that stops at the first failure has already run every other test; it
also passes on its own in a fresh process.
"""
import ctypes as C

import pytest
import torch

from block_sparse_attention_do_gb300 import api, inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_sparse_attention_do_gb300 import build

    build.build()
    api.lib()


def _problem(idx, Hq, bs, cu, max_seqlen):
    if cu is None:
        B, Hkv, T, S = idx.shape
        return api.problem(B, Hq, Hkv, T, 128, bs, S, torch.bfloat16), B * T
    total, Hkv, S = idx.shape
    return api.problem(cu.numel() - 1, Hq, Hkv, max_seqlen, 128, bs, S, torch.bfloat16,
                       layout=api.LAYOUT_THD, total_tokens=total), total


def _noalloc(idx, Hq, bs, cu=None, max_seqlen=None):
    """Calls the no-allocation entry point through the C ABI.  The test (the
    caller) owns the output buffers; the entry point allocates nothing."""
    p, ntok = _problem(idx, Hq, bs, cu, max_seqlen)
    L = api.lib()
    noff = int(L.nsa_inverse_index_offsets_len(C.byref(p)))
    offsets = torch.full((noff,), -7, dtype=torch.int32, device=DEV)
    rows = torch.full((max(1, ntok * idx.shape[-2] * idx.shape[-1]),), -7, dtype=torch.int32,
                      device=DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    s = L.nsa_build_inverse_index_noalloc(C.byref(p), api._ptr(cu), api._ptr(idx), api._ptr(offsets),
                                          api._ptr(rows), api._ptr(status), api._stream())
    return s, offsets, rows, status


def _cases():
    # a fixed-length problem with the long-sequence shape's block structure,
    # then a packed variable-length one: two different calls in a row
    a = inputs.make_block_idx(1, 2, 2048, 64, 16, seed=11)
    lengths = [300, 64, 1000, 17]
    b = inputs.make_varlen_block_idx(lengths, 4, 64, 8, seed=12)
    cu = inputs.cu_seqlens_from_lengths(lengths)
    return [(a, 32, 64, None, None), (b, 16, 64, cu, max(lengths))]


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    for idx, Hq, bs, cu, maxlen in _cases():
        gi = idx.to(DEV)
        gcu = None if cu is None else cu.to(DEV)
        ref_off, ref_rows, ws = api.build_inverse_index(gi, Hq, bs, cu_seqlens=gcu, max_seqlen=maxlen)
        s, off, rows, status = _noalloc(gi, Hq, bs, gcu, maxlen)
        assert s == api.NSA_OK
        torch.cuda.synchronize()
        n = int(ref_off[-1].item())
        assert torch.equal(off, ref_off)
        assert torch.equal(rows[:n], ref_rows[:n])
        assert int(status.item()) == api.NSA_OK
        assert api.get_error(ws) == api.NSA_OK


def test_noalloc_repeated_call_gives_identical_result():
    idx, Hq, bs, cu, maxlen = _cases()[0]
    gi = idx.to(DEV)
    first = _noalloc(gi, Hq, bs)
    second = _noalloc(gi, Hq, bs)
    torch.cuda.synchronize()
    assert first[0] == second[0] == api.NSA_OK
    assert torch.equal(first[1], second[1]) and torch.equal(first[2], second[2])


def test_noalloc_reports_bad_index_and_recovers():
    idx = inputs.make_block_idx(1, 1, 256, 64, 4, seed=3)
    bad = idx.clone()
    bad[0, 0, 10, 1] = 2  # a block in the future of token 10
    s, _, _, status = _noalloc(bad.to(DEV), 4, 64)
    torch.cuda.synchronize()
    assert s == api.NSA_OK and int(status.item()) == 3  # NSA_ERR_BAD_INDEX
    s, off, rows, status = _noalloc(idx.to(DEV), 4, 64)
    torch.cuda.synchronize()
    assert s == api.NSA_OK and int(status.item()) == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 64 x 64 kv heads x 1024 blocks = 4M per-block counters: far over 2 MiB
    p = api.problem(64, 64, 64, 65536, 128, 64, 16, torch.bfloat16)
    dummy = C.c_void_p(256)
    s = api.lib().nsa_build_inverse_index_noalloc(C.byref(p), None, dummy, dummy, dummy, None, None)
    assert s == 2  # NSA_ERR_UNSUPPORTED, returned before any launch
