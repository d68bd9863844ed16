#!/usr/bin/env python
"""Benchmark of the NSA block-selection attention hot path on GB300.

One step = one pass of the whole path over the workload: the selection
forward (O, LSE) and the backward (do_dot, inverse index, dK/dV, dQ), all
through the C ABI of libnsa.so.  The headline metric is the backward's
effective throughput: 10 * D FLOP per (query row, attended key) pair summed
over query heads (5 matmuls x 2 D), selected blocks only, divided by the time
of the whole nsa_sel_bwd call.

Workload: B=1, Hq=32, Hkv=2 (G=16), T=8192, D=128, block_size=64, S=16, bf16,
q/k/v/dO ~ N(0,1), each token selecting its own causal block plus 15 earlier
blocks drawn uniformly (seeded), as produced by
block_sparse_attention_do_gb300.inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs an independent replica (its own seed) of the
workload on its own GPU: the problems share nothing, so there is no
collective on the data path (weak scaling); rank 0 prints one JSON line.
`--impl reference` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NSA-selection bwd effective TFLOP/s (selected blocks only) and % of bf16 tensor peak"
WORKLOAD = dict(B=1, Hq=32, Hkv=2, T=8192, D=128, block_size=64, S=16)
WORKLOAD_NAME = ("NSA selection fwd+bwd, bf16: B=1 Hq=32 Hkv=2 (G=16) T=8192 D=128 "
                 "block_size=64 S=16, own block + 15 uniform earlier blocks per token")
# FLOP per selected (query row, key) pair of each kernel's algorithmic work
ALG_FLOP_PER_PAIR_PER_D = {"dkdv_tc": 8, "dq_tc": 6, "fwd_tc": 4,
                           "dkdv_gtc": 8, "dq_gtc": 6, "fwd_gtc": 4,
                           "dkdv_simt": 8, "dq_simt": 6, "fwd_simt": 4}
FLUSH_BYTES = 256 << 20  # > the 129 MB L2
SWA_WINDOW = 512  # sliding-window leg: keys (t - 512, t]


def env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def aggregate(local_time_ms: float, local_flop: float, device=None):
    """Max of the time and sum of the work over ranks (identity at N=1)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return local_time_ms, local_flop
    t = torch.tensor([local_time_ms], dtype=torch.float64, device=device)
    w = torch.tensor([local_flop], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(w, op=dist.ReduceOp.SUM)
    return float(t.item()), float(w.item())


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed loop runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        # the raw samples, beside the summary the JSON line carries
        out_dir = os.environ.get("NSA_BENCH_OUT") or os.path.join(ROOT, "bench_out")
        self.path = os.path.join(out_dir, f"clocks_rank{gpu_index}.csv")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    rows.append((float(parts[0]), float(parts[1]), parts[3:8]))
                except ValueError:
                    continue
        if not rows:
            return None
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for _, _, flags in rows:
            for n, v in zip(names[1:], flags[1:]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


def kernel_source_hash(name: str) -> str:
    files = {"dkdv_tc": "k_tc_dkdv.cu", "dq_tc": "k_tc_dq.cu", "fwd_tc": "k_tc_fwd.cu"}
    f = files.get(name)
    if f is None:
        return ""
    with open(os.path.join(ROOT, "block_sparse_attention_do_gb300", "csrc", f), "rb") as fh:
        return hashlib.sha256(fh.read()).hexdigest()[:16]


def traffic_for(name: str):
    """DRAM bytes per launch from the committed ncu summary, if it is current."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(name)
    if not e or e.get("source_sha") != kernel_source_hash(name):
        return None
    return e.get("bytes_per_launch_full")


def cpu_baseline_oracle(heads: int, T_prefix: int | None = None):
    """Time the fp64 oracle's backward on a bounded sample of the workload:
    kv group 0 of batch 0 with its first `heads` query heads (a self-contained
    sub-problem of the same selection), optionally the first T_prefix tokens."""
    import torch

    import oracle
    from block_sparse_attention_do_gb300 import inputs

    W = WORKLOAD
    T = W["T"] if T_prefix is None else T_prefix
    q, k, v, do = inputs.make_qkv_do(W["B"], W["Hq"], W["Hkv"], W["T"], W["D"], dtype=torch.bfloat16,
                                     seed=0)
    idx = inputs.make_block_idx(W["B"], W["Hkv"], W["T"], W["block_size"], W["S"], seed=0)
    q, do = q[:, :heads, :T], do[:, :heads, :T]
    k, v, idx = k[:, :1, :T], v[:, :1, :T], idx[:, :1, :T]
    pairs = oracle.count_pairs(idx, heads, W["block_size"])
    t0 = time.perf_counter()
    oracle.sel_bwd(q, k, v, idx, do, W["block_size"])
    dt = time.perf_counter() - t0
    cores = int(os.environ.get("OMP_NUM_THREADS", len(os.sched_getaffinity(0))))
    return dict(seconds=dt, pairs=pairs, flop=10 * W["D"] * pairs, cores=cores,
                sample=f"kv group 0, query heads 0..{heads - 1}, tokens 0..{T - 1} "
                       f"({pairs} pairs; fp64 backward incl. its forward recompute)")


def dense_pairs(B, Hq, T):
    """(query row, key) pairs of dense causal attention: every row t attends t + 1 keys."""
    return B * Hq * T * (T + 1) // 2


def bench_extra(name, q, k, v, do, idx, bs, flush, st, steps, peaks, cu=None, dense=False, pairs=None):
    """Times one more workload of the pages' configs through the C ABI: the
    backward (median of `steps`, L2 flushed before each) and the forward, then
    a traced pass for the per-kernel breakdown and the dominant kernel's
    roofline (its own algorithmic FLOPs per pair)."""
    import torch

    from block_sparse_attention_do_gb300 import api

    D, Hq = q.shape[-1], q.shape[-3] if cu is None else q.shape[1]
    if pairs is None:
        pairs = api.count_pairs(idx, Hq, bs, cu_seqlens=cu)
    flop = 10.0 * D * pairs
    gi = None if dense else idx
    o, lse = api.sel_fwd(q, k, v, gi, bs, cu_seqlens=cu, dense=dense)
    outs = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    for _ in range(3):
        o, lse = api.sel_fwd(q, k, v, gi, bs, cu_seqlens=cu, dense=dense)
        api.sel_bwd(q, k, v, o, do, lse, gi, bs, cu_seqlens=cu, dense=dense, out=outs)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        ev[i][0].record(st)
        o, lse = api.sel_fwd(q, k, v, gi, bs, cu_seqlens=cu, dense=dense)
        ev[i][1].record(st)
        api.sel_bwd(q, k, v, o, do, lse, gi, bs, cu_seqlens=cu, dense=dense, out=outs)
        ev[i][2].record(st)
    torch.cuda.synchronize()
    bwd = sorted(e[1].elapsed_time(e[2]) for e in ev)
    fwd = sorted(e[0].elapsed_time(e[1]) for e in ev)
    med_b, med_f = statistics.median(bwd), statistics.median(fwd)
    # traced pass: per-kernel times
    api.trace_enable(steps * 16)
    api.trace_reset()
    for i in range(steps):
        flush.zero_()
        o, lse = api.sel_fwd(q, k, v, gi, bs, cu_seqlens=cu, dense=dense)
        api.sel_bwd(q, k, v, o, do, lse, gi, bs, cu_seqlens=cu, dense=dense, out=outs)
    torch.cuda.synchronize()
    recs = api.trace_records()
    api.trace_enable(0)
    kern = {}
    for kn, ms in recs:
        e = kern.setdefault(kn, {"ms_total": 0.0, "launches": 0})
        e["ms_total"] += ms
        e["launches"] += 1
    bwd_kernels = {kn: e for kn, e in kern.items() if not kn.startswith("fwd")}
    for e in kern.values():
        e["ms_avg"] = e["ms_total"] / e["launches"]
    dom = max(bwd_kernels, key=lambda n: bwd_kernels[n]["ms_total"])
    roof = None
    if dom in ALG_FLOP_PER_PAIR_PER_D:
        alg = ALG_FLOP_PER_PAIR_PER_D[dom] * D * pairs
        ach = alg / (kern[dom]["ms_avg"] * 1e-3) / 1e12
        peak = float(peaks["bf16_tflops"])
        roof = {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "frac": ach / peak, "algorithmic_flop_per_launch": alg}
    return {"workload": name, "pairs": pairs, "bwd_flop": flop, "value": flop / (med_b * 1e-3) / 1e12,
            "unit": "TFLOP/s", "bwd_ms_median": med_b, "bwd_ms_mean": sum(bwd) / len(bwd),
            "fwd_ms_median": med_f, "steps": steps, "pct_of_bf16_peak": flop / (med_b * 1e-3) / 1e12 / float(
                peaks["bf16_tflops"]),
            "kernels": {kn: {"ms_avg": e["ms_avg"], "launches": e["launches"] // steps}
                        for kn, e in sorted(kern.items(), key=lambda kv: -kv[1]["ms_total"])},
            "roofline": roof}


def run_reference(args):
    rank, _, world = env_rank()
    if rank != 0:
        return 0
    import oracle

    oracle.build()
    # one step = the oracle's backward on the same kind of sample as the
    # cpu_baseline key of the GPU arm (kv group 0, the first `heads` query
    # heads, full length), with as many heads as fit about 150 s for the run
    budget = min(12.0, 150.0 / (args.steps + args.warmup))
    cal = cpu_baseline_oracle(1)
    heads = max(1, min(16, int(budget / cal["seconds"])))
    for _ in range(max(0, args.warmup - 1)):
        cpu_baseline_oracle(heads)
    secs, flop = 0.0, 0.0
    last = None
    for _ in range(args.steps):
        r = cpu_baseline_oracle(heads)
        secs += r["seconds"]
        flop += r["flop"]
        last = r
    value = flop / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, **WORKLOAD, "parallelism": "host cores (OpenMP)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": last["cores"], "kind": "oracle",
                         "sample": last["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, local_rank, world = env_rank()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    from block_sparse_attention_do_gb300 import api, build, inputs

    build.build()
    W = WORKLOAD
    B, Hq, Hkv, T, D, bs, S = (W[k] for k in ("B", "Hq", "Hkv", "T", "D", "block_size", "S"))
    q, k, v, do = inputs.make_qkv_do(B, Hq, Hkv, T, D, dtype=torch.bfloat16, seed=rank)
    idx = inputs.make_block_idx(B, Hkv, T, bs, S, seed=rank)
    q, k, v, do, idx = (x.to(dev) for x in (q, k, v, do, idx))
    pairs = api.count_pairs(idx, Hq, bs)
    bwd_flop = 10.0 * D * pairs

    p = api.problem_from(q, k, bs, S)
    ws_f = torch.empty(api.fwd_workspace_size(p), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(api.bwd_workspace_size(p), dtype=torch.uint8, device=dev)
    outs = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream()

    def step():
        o, lse = api.sel_fwd(q, k, v, idx, bs, ws=ws_f)
        return o, lse

    for _ in range(args.warmup):
        o, lse = step()
        api.sel_bwd(q, k, v, o, do, lse, idx, bs, ws=ws_b, out=outs)
    torch.cuda.synchronize()
    if api.get_error(ws_b) != 0 or api.get_error(ws_f) != 0:
        raise RuntimeError("device error during warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(local_rank)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(K):
        flush.zero_()  # evict L2 between steps (outside the timed events)
        ev[i][0].record(st)
        o, lse = api.sel_fwd(q, k, v, idx, bs, ws=ws_f)
        ev[i][1].record(st)
        api.sel_bwd(q, k, v, o, do, lse, idx, bs, ws=ws_b, out=outs)
        ev[i][2].record(st)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = sum(e[1].elapsed_time(e[2]) for e in ev)
    step_ms = sum(e[0].elapsed_time(e[2]) for e in ev)
    # the median of the K backward times (the headline) beside the mean
    bwd_med = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    err = api.get_error(ws_b) or api.get_error(ws_f)
    if err:
        raise RuntimeError(f"device error status {err} in the timed loop")

    # ---- per-kernel times: a second pass of the same K steps with the
    # library's per-launch event tracer on.  Its event records sit between
    # the launches, which also stops a kernel from starting while the one
    # before it drains, so the headline above is timed without them.
    api.trace_enable(K * 16)
    api.trace_reset()
    tr_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush.zero_()
        o, lse = api.sel_fwd(q, k, v, idx, bs, ws=ws_f)
        tr_ev[i][0].record(st)
        api.sel_bwd(q, k, v, o, do, lse, idx, bs, ws=ws_b, out=outs)
        tr_ev[i][1].record(st)
    torch.cuda.synchronize()
    recs = api.trace_records()
    api.trace_enable(0)
    traced_bwd_ms = sum(a.elapsed_time(b) for a, b in tr_ev) / K

    bwd_ms_max, flop_all = aggregate(bwd_ms, bwd_flop * K, dev)
    med_max, flop_one = aggregate(bwd_med, bwd_flop, dev)
    step_ms_max, _ = aggregate(step_ms, 0.0, dev)
    value = flop_one / (med_max * 1e-3) / 1e12
    value_mean = flop_all / (bwd_ms_max * 1e-3) / 1e12

    # ---- per-kernel breakdown and roofline of the dominant kernel
    kern = {}
    for name, ms in recs:
        e = kern.setdefault(name, {"ms_total": 0.0, "launches": 0})
        e["ms_total"] += ms
        e["launches"] += 1
    total_k = sum(e["ms_total"] for e in kern.values()) or 1.0
    for name, e in kern.items():
        e["ms_avg"] = e["ms_total"] / e["launches"]
        e["share"] = e["ms_total"] / total_k
    peaks, peak_src = load_peaks()
    dom = max(kern, key=lambda n: kern[n]["ms_total"])
    roof = None
    if dom in ALG_FLOP_PER_PAIR_PER_D:
        alg = ALG_FLOP_PER_PAIR_PER_D[dom] * D * pairs
        ach = alg / (kern[dom]["ms_avg"] * 1e-3) / 1e12
        peak = float(peaks["bf16_tflops"])
        roof = {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "frac": ach / peak, "traffic": traffic_for(dom),
                "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json bf16_tflops)",
                "algorithmic_flop_per_launch": alg}
    pct = value / float(peaks["bf16_tflops"])

    # ---- the same backward reading a plan built once for idx (nsa_plan_build):
    # the inverse index leaves the backward's critical path
    plan_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    plan_ev[0].record(st)
    plan = api.build_plan(q, k, idx, bs)
    plan_ev[1].record(st)
    ws_p = torch.empty(api.bwd_planned_workspace_size(p), dtype=torch.uint8, device=dev)
    o, lse = step()
    for _ in range(2):
        api.sel_bwd(q, k, v, o, do, lse, idx, bs, ws=ws_p, out=outs, plan=plan)
    n_pl = max(3, min(K, 50))
    p_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_pl)]
    for i in range(n_pl):
        flush.zero_()
        p_ev[i][0].record(st)
        api.sel_bwd(q, k, v, o, do, lse, idx, bs, ws=ws_p, out=outs, plan=plan)
        p_ev[i][1].record(st)
    torch.cuda.synchronize()
    if api.get_error(ws_p) or api.get_error(plan):
        raise RuntimeError("device error in the planned backward")
    pl_ms = sum(a.elapsed_time(b) for a, b in p_ev)
    pl_ms_max, pl_flop = aggregate(pl_ms, bwd_flop * n_pl, dev)
    planned = {"value": pl_flop / (pl_ms_max * 1e-3) / 1e12, "unit": "TFLOP/s", "bwd_ms": pl_ms / n_pl,
               "plan_build_ms": plan_ev[0].elapsed_time(plan_ev[1]), "steps": n_pl,
               "scope": "nsa_sel_bwd_planned with a plan built once for idx (nsa_plan_build, timed "
                        "apart); same L2 flush between steps"}

    # ---- sliding-window causal attention (nsa_swa_fwd / nsa_swa_bwd) on the
    # same tensors: every row attends its SWA_WINDOW most recent keys
    Wn = SWA_WINDOW
    swa_pairs = B * Hq * sum(min(t + 1, Wn) for t in range(T))
    o_w, lse_w = api.sel_fwd(q, k, v, None, bs, window=Wn, ws=ws_f)
    for _ in range(2):
        api.sel_bwd(q, k, v, o_w, do, lse_w, None, bs, window=Wn, ws=ws_b, out=outs)
    n_sw = max(3, min(K, 20))
    w_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_sw)]
    for i in range(n_sw):
        flush.zero_()
        w_ev[i][0].record(st)
        o_w, lse_w = api.sel_fwd(q, k, v, None, bs, window=Wn, ws=ws_f)
        w_ev[i][1].record(st)
        api.sel_bwd(q, k, v, o_w, do, lse_w, None, bs, window=Wn, ws=ws_b, out=outs)
        w_ev[i][2].record(st)
    torch.cuda.synchronize()
    if api.get_error(ws_b) or api.get_error(ws_f):
        raise RuntimeError("device error in the sliding-window leg")
    sw_bwd = sum(e[1].elapsed_time(e[2]) for e in w_ev)
    sw_fwd = sum(e[0].elapsed_time(e[1]) for e in w_ev)
    sw_bwd_max, sw_flop = aggregate(sw_bwd, 10.0 * D * swa_pairs * n_sw, dev)
    swa = {"window": Wn, "pairs": swa_pairs, "value": sw_flop / (sw_bwd_max * 1e-3) / 1e12, "unit": "TFLOP/s",
           "bwd_ms": sw_bwd / n_sw, "fwd_ms": sw_fwd / n_sw, "steps": n_sw,
           "scope": "nsa_swa_fwd + nsa_swa_bwd, same shapes, 10*D*pairs / backward time, L2 flushed"}

    # ---- the step that produces the index (nsa_compress_keys_mean,
    # nsa_block_scores, nsa_select_topk) on the same q and k: compressed keys,
    # block scores on the tensor cores, the own block + S-1 best complete blocks
    kc = api.compress_keys_mean(k, bs)
    for _ in range(2):
        sc_ = api.block_scores(q, kc, bs)
        api.select_topk(sc_, bs, S)
    n_se = max(3, min(K, 20))
    s_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_se)]
    for i in range(n_se):
        flush.zero_()
        # the three calls are short: a ~0.1 ms wait queued first lets the host
        # enqueue them all, so the events time the GPU rather than the launches
        torch.cuda._sleep(200_000)
        s_ev[i][0].record(st)
        kc = api.compress_keys_mean(k, bs)
        s_ev[i][1].record(st)
        sc_ = api.block_scores(q, kc, bs)
        s_ev[i][2].record(st)
        idx_sel = api.select_topk(sc_, bs, S)
        s_ev[i][3].record(st)
    torch.cuda.synchronize()
    if api.get_error(api.workspace(1, dev, "select")):
        raise RuntimeError("device error in the selection-step leg")
    sel_ms = [sorted(e[j].elapsed_time(e[j + 1]) for e in s_ev)[n_se // 2] for j in range(3)]
    nb_sel = (T + bs - 1) // bs
    esz = 2
    sc_bytes = B * Hq * T * D * esz + B * Hkv * nb_sel * D * esz + B * Hkv * T * nb_sel * 4
    peak_hbm = peaks.get("hbm_gbs") if peaks else None
    select = {
        "ms": {"compress_mean": sel_ms[0], "block_scores": sel_ms[1], "select_topk": sel_ms[2]},
        "step_ms": sum(sel_ms), "steps": n_se, "index_rows": B * Hkv * T,
        "rows_per_s": B * Hkv * T / (sum(sel_ms) * 1e-3),
        "roofline": {"kernel": "block_scores", "bound": "hbm", "unit": "GB/s",
                     "achieved": sc_bytes / (sel_ms[1] * 1e-3) / 1e9, "peak": peak_hbm,
                     "frac": (sc_bytes / (sel_ms[1] * 1e-3) / 1e9 / peak_hbm) if peak_hbm else None,
                     "algorithmic_bytes": sc_bytes,
                     "bytes_are": "read q and kc once, write fp32 scores [B,Hkv,T,nb] once"},
        "scope": "median per kernel over the steps, L2 flushed before each step, the calls queued behind a "
                 "GPU wait so that host launch time is not counted; same q and k as the headline",
    }
    del kc, sc_, idx_sel

    # ---- the pages' other workloads (single GPU only; rank 0 of a replica run
    # times them too, each rank on its own GPU)
    configs = {}
    if not args.skip_configs:
        n_x = max(5, min(K, 20))
        # config 2 in bf16: B=2 Hq=6 Hkv=2 T=1024 D=64 block 32 S=8
        q2, k2, v2, do2 = inputs.make_qkv_do(2, 6, 2, 1024, 64, dtype=torch.bfloat16, seed=rank)
        idx2 = inputs.make_block_idx(2, 2, 1024, 32, 8, seed=rank)
        configs["mid_bf16"] = bench_extra(
            "NSA selection bwd, bf16: B=2 Hq=6 Hkv=2 (G=3) T=1024 D=64 block_size=32 S=8",
            *(x.to(dev) for x in (q2, k2, v2, do2, idx2)), 32, flush, st, n_x, peaks)
        # ... and in fp32 (split precision: three bf16 products per fp32 product;
        # the roofline still counts the fp32 work against the bf16 peak)
        q2, k2, v2, do2 = inputs.make_qkv_do(2, 6, 2, 1024, 64, dtype=torch.float32, seed=rank)
        configs["mid_fp32"] = bench_extra(
            "NSA selection bwd, fp32: B=2 Hq=6 Hkv=2 (G=3) T=1024 D=64 block_size=32 S=8",
            *(x.to(dev) for x in (q2, k2, v2, do2, idx2)), 32, flush, st, n_x, peaks)
        del q2, k2, v2, do2, idx2
        # config 4: dense causal B=2 Hq=32 Hkv=8 T=4096 D=128 block 64 (nsa_dense_causal_*)
        q4, k4, v4, do4 = inputs.make_qkv_do(2, 32, 8, 4096, 128, dtype=torch.bfloat16, seed=rank)
        configs["dense_causal"] = bench_extra(
            "dense causal SDPA bwd as selection of all valid blocks, bf16: B=2 Hq=32 Hkv=8 (G=4) T=4096 "
            "D=128 block_size=64", *(x.to(dev) for x in (q4, k4, v4, do4)), None, 64, flush, st, n_x, peaks,
            dense=True, pairs=dense_pairs(2, 32, 4096))
        del q4, k4, v4, do4
        # config 5: THD, 8 sequences with lengths uniform in [128, 4096], Hq=32 Hkv=8 D=128 block 64 S=16
        lens = inputs.make_varlen_lengths(8, 128, 4096, seed=rank)
        cu5 = inputs.cu_seqlens_from_lengths(lens)
        q5, k5, v5, do5 = inputs.make_qkv_do(1, 32, 8, sum(lens), 128, dtype=torch.bfloat16, seed=rank,
                                             layout="thd")
        idx5 = inputs.make_varlen_block_idx(lens, 8, 64, 16, seed=rank)
        configs["varlen_thd"] = bench_extra(
            f"THD varlen NSA selection bwd, bf16: 8 sequences (lengths {lens}), Hq=32 Hkv=8 (G=4) D=128 "
            "block_size=64 S=16", *(x.to(dev) for x in (q5, k5, v5, do5, idx5)), 64, flush, st, n_x, peaks,
            cu=cu5.to(dev))
        del q5, k5, v5, do5, idx5
        torch.cuda.synchronize()
        if api.get_error(api.workspace(1, dev, "bwd")) or api.get_error(api.workspace(1, dev, "fwd")):
            raise RuntimeError("device error in the extra workloads")

    # ---- end to end through the public API with host buffers
    e2e = None
    if True:  # every rank: the aggregation below is collective
        o, lse = step()
        torch.cuda.synchronize()
        host_in = [x.cpu().pin_memory() for x in (q, k, v, o, do, lse, idx)]
        dev_in = [torch.empty_like(x, device=dev) for x in host_in]
        host_out = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in outs]
        h2d = sum(x.numel() * x.element_size() for x in host_in)
        d2h = sum(x.numel() * x.element_size() for x in host_out)
        n_e2e = max(3, min(K, 20))
        # (1) one step at a time on one stream: copy in, backward, copy out
        e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(n_e2e + 2)]
        for i in range(n_e2e + 2):
            e_ev[i][0].record(st)
            for hsrc, ddst in zip(host_in, dev_in):
                ddst.copy_(hsrc, non_blocking=True)
            api.sel_bwd(*dev_in[:6], dev_in[6], bs, ws=ws_b, out=outs)
            for dsrc, hdst in zip(outs, host_out):
                hdst.copy_(dsrc, non_blocking=True)
            e_ev[i][1].record(st)
        torch.cuda.synchronize()
        serial_ms = sum(a.elapsed_time(b) for a, b in e_ev[2:]) / n_e2e  # first two are warm-up
        # (2) the same steps as a pipeline: step i's inputs go in on a copy
        # stream while step i-1 computes and step i-2's gradients come out on
        # another; two sets of device buffers alternate.  Every step still
        # copies all its inputs in and its gradients out inside the timed region.
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        dev_in2 = [dev_in, [torch.empty_like(x) for x in dev_in]]
        outs2 = [list(outs), [torch.empty_like(x) for x in outs]]
        host_out2 = [host_out, [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in outs]]

        def pipeline(n):
            done_c = [None, None]  # per buffer set: the compute that last read / wrote it
            done_o = [None, None]  # per buffer set: the copy-out that last read its gradients
            for i in range(n):
                j = i % 2
                ev_in = torch.cuda.Event()
                with torch.cuda.stream(s_in):
                    if done_c[j] is not None:
                        s_in.wait_event(done_c[j])
                    for hsrc, ddst in zip(host_in, dev_in2[j]):
                        ddst.copy_(hsrc, non_blocking=True)
                    ev_in.record(s_in)
                st.wait_event(ev_in)
                if done_o[j] is not None:
                    st.wait_event(done_o[j])
                api.sel_bwd(*dev_in2[j][:6], dev_in2[j][6], bs, ws=ws_b, out=outs2[j])
                done_c[j] = torch.cuda.Event()
                done_c[j].record(st)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done_c[j])
                    for dsrc, hdst in zip(outs2[j], host_out2[j]):
                        hdst.copy_(dsrc, non_blocking=True)
                    done_o[j] = torch.cuda.Event()
                    done_o[j].record(s_out)
            st.wait_stream(s_in)
            st.wait_stream(s_out)

        pipeline(2)
        torch.cuda.synchronize()
        p_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        p_ev[0].record(st)
        s_in.wait_stream(st)
        s_out.wait_stream(st)
        pipeline(n_e2e)
        p_ev[1].record(st)
        torch.cuda.synchronize()
        if api.get_error(ws_b):
            raise RuntimeError("device error in the end-to-end leg")
        e_ms = p_ev[0].elapsed_time(p_ev[1])
        e_ms_max, e_flop = aggregate(e_ms, bwd_flop * n_e2e, dev)
        e2e = {"value": e_flop / (e_ms_max * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms / n_e2e, "steps": n_e2e,
               "serial_ms_per_step": serial_ms,
               "scope": "per step: H2D of the backward's inputs (q,k,v,o,dO,lse,idx) from pinned memory, "
                        "nsa_sel_bwd, D2H of dq,dk,dv to pinned memory; steps pipelined over a copy-in "
                        "stream, the compute stream and a copy-out stream with two buffer sets "
                        "(serial_ms_per_step: the same step alone on one stream)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = cpu_baseline_oracle(args.cpu_heads)
        cpu = {"value": r["flop"] / r["seconds"] / 1e12, "unit": "TFLOP/s", "cores": r["cores"],
               "kind": "oracle", "sample": r["sample"], "seconds": r["seconds"],
               "note": "the stated CPU baseline; bench.py --impl reference times the same kind of sample "
                       "(fewer heads per step)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": step_ms_max / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD_NAME, **WORKLOAD, "pairs": pairs,
                       "bwd_flop_per_step": bwd_flop,
                       "l2": "flushed between steps (256 MiB write outside the timed events); "
                             "the bwd also reads 192 MiB of q/o/dO, more than L2",
                       "parallelism": f"replicas x{world} (independent problems, no collective)"},
            "pct_of_bf16_peak": pct,
            "value_is": "10*D*pairs / median backward time over the K timed steps",
            "value_mean": value_mean,
            "bwd_ms": bwd_med, "bwd_ms_mean": bwd_ms / K, "fwd_ms": fwd_ms / K, "wall_s": t_wall,
            "kernels": {n: {"ms_avg": e["ms_avg"], "launches": e["launches"], "share": e["share"]}
                        for n, e in sorted(kern.items(), key=lambda kv: -kv[1]["ms_total"])},
            "kernels_pass": {"what": "a second pass of the same K fwd+bwd steps with a CUDA event pair "
                                     "around every launch (the library's tracer); the roofline uses it",
                             "bwd_ms": traced_bwd_ms},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "planned": planned, "swa": swa,
            "select": select,
            "configs": configs,
            "gpu_launches": len(recs),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-heads", type=int, default=4, help="query heads in the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-configs", action="store_true", help="time only the headline workload")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
