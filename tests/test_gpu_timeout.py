"""The tensor-core kernels' bounded waits, run out on purpose without any
fault: nsa_debug_stall keeps one kernel's S-product issuer idle and shortens
every wait to a few milliseconds.  The kernel must then stop, wait for its
own copies and products in flight, free its tensor memory and report
NSA_ERR_DEVICE_TIMEOUT through the workspace error word; the next normal call
on the same stream must run and match the oracle (the context is usable and
tensor memory was released)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_do_gb300 import api, inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "gate_tolerances.json")))
TOL = GOLD["max_abs_gate"]["bf16"]
TIMEOUT = 4  # NSA_ERR_DEVICE_TIMEOUT


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_sparse_attention_do_gb300 import build

    build.build()
    api.lib()
    yield
    api.debug_stall(0, 0)


def _problem():
    # the tensor-core path: bf16, D = 128, 64-key blocks, G = 16, a ragged end
    B, Hq, Hkv, T, D, bs, S = 1, 16, 1, 700, 128, 64, 4
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.bfloat16, seed=31)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=31)
    return (q, k, v, do, idx), bs


def _check_normal(cpu, g, bs, ws_f, ws_b):
    q, k, v, do, idx = cpu
    o, lse = api.sel_fwd(g[0], g[1], g[2], g[4], bs, ws=ws_f)
    dq, dk, dv = api.sel_bwd(g[0], g[1], g[2], o, g[3], lse, g[4], bs, ws=ws_b)
    torch.cuda.synchronize()
    assert api.get_error(ws_f) == 0 and api.get_error(ws_b) == 0
    ref = oracle.sel_bwd(q, k, v, idx, do, bs)
    for name, x in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        err = float(np.max(np.abs(x.double().cpu().numpy() - ref[name]) - 2.0 ** -8 * np.abs(ref[name])))
        assert err <= TOL, (name, err)


@pytest.mark.parametrize("kernel", [1, 2, 3], ids=["forward", "dkdv", "dq"])
def test_wait_runs_out_reports_timeout_and_recovers(kernel):
    cpu, bs = _problem()
    g = [x.to(DEV) for x in cpu]
    p = api.problem_from(g[0], g[1], bs, cpu[4].shape[-1])
    ws_f = torch.empty(api.fwd_workspace_size(p), dtype=torch.uint8, device=DEV)
    ws_b = torch.empty(api.bwd_workspace_size(p), dtype=torch.uint8, device=DEV)
    # a normal forward first: the backward below needs its o and lse
    o, lse = api.sel_fwd(g[0], g[1], g[2], g[4], bs, ws=ws_f)
    torch.cuda.synchronize()
    assert api.get_error(ws_f) == 0
    api.debug_stall(kernel, 5000)  # 5 ms waits
    try:
        if kernel == 1:
            api.sel_fwd(g[0], g[1], g[2], g[4], bs, ws=ws_f)
            ws = ws_f
        else:
            api.sel_bwd(g[0], g[1], g[2], o, g[3], lse, g[4], bs, ws=ws_b)
            ws = ws_b
        torch.cuda.synchronize()  # the launch returned: every wait ended
    finally:
        api.debug_stall(0, 0)
    assert api.get_error(ws) == TIMEOUT
    assert api.get_error(ws) == 0  # reading clears it
    # the same stream and context, normal operation: parity with the oracle
    _check_normal(cpu, g, bs, ws_f, ws_b)
