"""The C ABI library loads on a machine without a GPU and exports every
function include/nsa.h declares; host-side argument checks return the
documented statuses without touching a device."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_sparse_attention_do_gb300 import api, build

    build.build()
    return api.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "nsa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nsa_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    from block_sparse_attention_do_gb300 import api

    declared = _declared()
    assert len(declared) >= 14
    assert sorted(api.SYMBOLS) == declared
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.nsa_status_string(0) == b"NSA_OK"
    assert lib.nsa_status_string(3) == b"NSA_ERR_BAD_INDEX"
    assert lib.nsa_status_string(99) == b"NSA_ERR_UNKNOWN"


def _p(**kw):
    import torch

    from block_sparse_attention_do_gb300 import api

    base = dict(B=1, Hq=4, Hkv=2, T=256, D=128, block_size=64, S=4, dtype=torch.bfloat16)
    base.update(kw)
    return api.problem(**base)


def test_workspace_sizes_and_validation(lib):
    from block_sparse_attention_do_gb300 import api

    p = _p()
    assert api.fwd_workspace_size(p) >= 256
    assert lib.nsa_sel_fwd_workspace_size(C.byref(p)) == api.fwd_workspace_size(p)
    assert lib.nsa_sel_bwd_workspace_size(C.byref(p)) == api.bwd_workspace_size(p)
    assert api.bwd_workspace_size(p) > 256 + 4 * 256 * 4
    assert api.bwd_workspace_size(_p(Hq=3)) == 0          # Hq % Hkv != 0
    assert api.bwd_workspace_size(_p(D=96)) == 0          # unsupported head dim
    assert api.bwd_workspace_size(_p(block_size=48)) == 0
    # a call with null tensors fails before any launch
    ws = C.c_void_p(256)
    s = lib.nsa_sel_fwd(C.byref(p), None, None, None, None, None, None, ws, 1 << 20, None)
    assert s == 1
    s = lib.nsa_sel_bwd(C.byref(_p(D=96)), *([C.c_void_p(256)] * 10), ws, 1 << 20, None)
    assert s == 2
    # workspace too small / misaligned
    args = [C.c_void_p(256)] * 6
    assert lib.nsa_sel_fwd(C.byref(p), *args, C.c_void_p(256), 16, None) == 6
    assert lib.nsa_sel_fwd(C.byref(p), *args, C.c_void_p(272), 1 << 20, None) == 6
    # misaligned tensor
    bad = [C.c_void_p(258)] + [C.c_void_p(256)] * 5
    assert lib.nsa_sel_fwd(C.byref(p), *bad, C.c_void_p(256), 1 << 20, None) == 1
    # wrong layout for the entry point
    pt = api.problem(1, 4, 2, 256, 128, 64, 4, __import__("torch").bfloat16, layout=1,
                     total_tokens=256)
    assert lib.nsa_sel_fwd(C.byref(pt), *args, C.c_void_p(256), 1 << 20, None) == 1


def test_offsets_len(lib):
    assert lib.nsa_inverse_index_offsets_len(C.byref(_p(B=2, Hkv=2, T=130, block_size=64))) == 2 * 2 * 3 + 1


def test_forward_workspace_holds_the_union_table(lib):
    """The selection forward's workspace: a 256-byte header, then (bf16 on the
    tensor-core kernels) one union record per 128-row query tile: 12 header
    ints, a block bitmap per token, the union bitmap (words rounded up to 4)
    and the block list (rounded up to 4 ints), 128-byte rounded."""
    import torch

    from block_sparse_attention_do_gb300 import api

    def expected(B, Hq, Hkv, T, bs):
        G, nb = Hq // Hkv, -(-T // bs)
        words = -(-nb // 32)
        tq = 128 // G
        ints = 12 + tq * words + (words + 3) // 4 * 4 + (nb + 3) // 4 * 4
        rec = -(-ints * 4 // 128) * 128
        table = B * Hkv * -(-T // tq) * rec
        return 256 + -(-table // 256) * 256

    for B, Hq, Hkv, T in ((1, 32, 2, 8192), (2, 16, 1, 1100), (1, 64, 4, 65536)):
        p = _p(B=B, Hq=Hq, Hkv=Hkv, T=T, S=16)
        assert api.fwd_workspace_size(p) == expected(B, Hq, Hkv, T, 64), (B, Hq, Hkv, T)
        # the backward's workspace carries the same table besides its own parts
        assert api.bwd_workspace_size(p) > api.fwd_workspace_size(p)
    # the CUDA-core kernels build no table
    assert api.fwd_workspace_size(_p(dtype=torch.float32)) == 256
    assert api.fwd_workspace_size(_p(D=64)) == 256


def test_index_sizes_beyond_int32_are_refused(lib):
    """Inverse-index entries (tokens x kv heads x slots) are counted in int32:
    a problem one slot past that limit is refused before any launch, the one
    just inside it is accepted."""
    from block_sparse_attention_do_gb300 import api

    T = 1 << 24  # 16M tokens, 8 kv heads: 16 slots give 2^31 entries
    inside = _p(B=1, Hq=8, Hkv=8, T=T, D=32, block_size=64, S=15)
    over = _p(B=1, Hq=8, Hkv=8, T=T, D=32, block_size=64, S=16)
    assert lib.nsa_plan_size(C.byref(inside)) > 0
    assert lib.nsa_plan_size(C.byref(over)) == 0
    dummy = C.c_void_p(256)
    s = lib.nsa_sel_bwd(C.byref(over), *([dummy] * 10), dummy, 1 << 40, None)
    assert s == 2  # NSA_ERR_UNSUPPORTED


def test_debug_stall_checks_its_arguments(lib):
    assert lib.nsa_debug_stall(4, 0) == 1
    assert lib.nsa_debug_stall(1, -1) == 1
    assert lib.nsa_debug_stall(2, 3000000) == 1
    assert lib.nsa_debug_stall(0, 0) == 0


def test_noalloc_status_pointer_alignment(lib):
    from block_sparse_attention_do_gb300 import api

    p = _p(B=1, Hkv=1, T=256, S=4)
    dummy = C.c_void_p(256)
    s = lib.nsa_build_inverse_index_noalloc(C.byref(p), None, dummy, dummy, dummy, C.c_void_p(258), None)
    assert s == 1  # NSA_ERR_INVALID_ARG: status_out not 4-byte aligned


def test_declared_strides_are_checked(lib):
    """Strides must be positive multiples of 16 bytes; all-zero strides mean
    the dense layout (the other tests pass zero-initialised problems)."""
    from block_sparse_attention_do_gb300 import api

    p = _p()
    n_dense = api.bwd_workspace_size(p)
    assert n_dense > 0
    args = [C.c_void_p(256)] * 6
    ws = C.c_void_p(256)
    # a token stride of D + 1 bf16 elements: not a 16-byte multiple
    p.q_stride[:] = (4 * 256 * 129, 256 * 129, 129)
    assert lib.nsa_sel_fwd(C.byref(p), *args, ws, 1 << 30, None) == 1
    assert api.bwd_workspace_size(p) == 0
    # a zero head stride among non-zero ones
    p.q_stride[:] = (4 * 256 * 128, 0, 128)
    assert lib.nsa_sel_fwd(C.byref(p), *args, ws, 1 << 30, None) == 1
    # the dense strides written out equal the zero default
    p.q_stride[:] = (4 * 256 * 128, 256 * 128, 128)
    assert api.bwd_workspace_size(p) == n_dense
    # THD ignores the batch entry
    pt = api.problem(2, 4, 2, 256, 128, 64, 4, __import__("torch").bfloat16, layout=1, total_tokens=300)
    pt.kv_stride[:] = (7, 128, 4 * 128)
    assert api.fwd_workspace_size(pt) > 0
    pt.kv_stride[:] = (0, 129, 4 * 128)
    assert api.fwd_workspace_size(pt) == 0
    assert lib.nsa_sel_varlen_fwd(C.byref(pt), C.c_void_p(256), *([C.c_void_p(256)] * 6), ws, 1 << 30,
                                  None) == 1


def test_causal_entries_check_their_arguments(lib):
    """nsa_causal_*: the key geometry is validated before any launch."""
    from block_sparse_attention_do_gb300 import api

    p = _p(T=256)
    p.Tk = 300
    p.bottom_right = 1
    n = lib.nsa_causal_bwd_workspace_size(C.byref(p))
    assert n > 0
    assert lib.nsa_causal_fwd_workspace_size(C.byref(p)) >= 256
    p.bottom_right = 2
    assert lib.nsa_causal_bwd_workspace_size(C.byref(p)) == 0
    p.bottom_right = 0
    p.Tk = -1
    assert lib.nsa_causal_bwd_workspace_size(C.byref(p)) == 0
    # packed layout: both cu_seqlens or neither, and total_keys >= 1
    pt = api.problem(2, 4, 2, 256, 128, 64, 4, __import__("torch").bfloat16, layout=1, total_tokens=300)
    assert lib.nsa_causal_bwd_workspace_size(C.byref(pt)) == 0  # total_keys = 0
    pt.total_keys = 400
    pt.Tk = 256
    assert lib.nsa_causal_bwd_workspace_size(C.byref(pt)) > 0
    dummy = C.c_void_p(256)
    s = lib.nsa_causal_fwd(C.byref(pt), 0, dummy, None, *([dummy] * 5), dummy, 1 << 30, None)
    assert s == 1
    s = lib.nsa_causal_fwd(C.byref(p), -1, None, None, *([dummy] * 5), dummy, 1 << 30, None)
    assert s == 1


def test_selection_step_argument_checks(lib):
    """The selection-step entries (block scores, top-S, compressed keys)
    refuse bad arguments before any launch."""
    import torch

    from block_sparse_attention_do_gb300 import api

    p = _p()
    assert lib.nsa_select_workspace_size(C.byref(p)) == 256
    assert lib.nsa_select_workspace_size(C.byref(_p(Hq=3))) == 0       # Hq % Hkv != 0
    assert lib.nsa_select_workspace_size(C.byref(_p(D=96))) == 0       # unsupported head dim
    pt = api.problem(2, 4, 2, 256, 64, 32, 4, torch.bfloat16, layout=1, total_tokens=300)
    assert lib.nsa_select_workspace_size(C.byref(pt)) == 256           # THD sizes need no cu_seqlens
    dev = C.c_void_p(256)
    ws = C.c_void_p(256)
    # null / misaligned tensors
    assert lib.nsa_compress_keys_mean(C.byref(p), None, None, dev, None) == 1
    assert lib.nsa_compress_keys_mean(C.byref(p), None, C.c_void_p(258), dev, None) == 1
    assert lib.nsa_block_scores(C.byref(p), None, dev, dev, None, ws, 256, None) == 1
    assert lib.nsa_block_scores(C.byref(p), None, dev, dev, C.c_void_p(258), ws, 256, None) == 1
    assert lib.nsa_select_topk(C.byref(p), None, dev, None, None) == 1
    assert lib.nsa_select_topk(C.byref(p), None, C.c_void_p(257), dev, None) == 1
    # workspace too small or misaligned
    assert lib.nsa_block_scores(C.byref(p), None, dev, dev, dev, ws, 16, None) == 6
    assert lib.nsa_block_scores(C.byref(p), None, dev, dev, dev, C.c_void_p(272), 256, None) == 6
    # shapes: block size, head dim, S
    assert lib.nsa_block_scores(C.byref(_p(block_size=48)), None, dev, dev, dev, ws, 256, None) == 2
    assert lib.nsa_select_topk(C.byref(_p(S=0)), None, dev, dev, None) == 1
    assert lib.nsa_select_topk(C.byref(_p(S=300)), None, dev, dev, None) == 2
    # THD without cu_seqlens
    assert lib.nsa_select_topk(C.byref(pt), None, dev, dev, None) == 1
