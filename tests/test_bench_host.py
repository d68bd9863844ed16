"""Host-side logic of bench.py: the multi-rank aggregation (max of time, sum
of work) over a world-size-2 gloo group on CPU, the reference arm's rank
handling, and the DRAM-traffic figure taken from the committed profile only
while it matches the kernel's source."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t, w = bench.aggregate(10.0 + rank * 5.0, 100.0 * (rank + 1), device="cpu")
    out[rank] = (t, w)
    dist.destroy_process_group()


def test_aggregate_gloo_world2():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1] == (15.0, 300.0)


def test_aggregate_single_process_is_identity():
    import bench

    assert bench.aggregate(3.0, 7.0) == (3.0, 7.0)


def test_reference_arm_nonzero_rank_exits_without_work(monkeypatch):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0


@pytest.mark.parametrize("argv", [["--warmup", "2"]])
def test_warmup_floor(argv):
    import bench

    with pytest.raises(SystemExit):
        bench.main(argv)


def test_traffic_only_for_the_profiled_source(tmp_path, monkeypatch):
    import json
    import shutil

    import bench

    src = os.path.join(bench.ROOT, "block_sparse_attention_do_gb300", "csrc", "k_tc_dkdv.cu")
    os.makedirs(tmp_path / "profiles")
    os.makedirs(tmp_path / "block_sparse_attention_do_gb300" / "csrc")
    shutil.copy(src, tmp_path / "block_sparse_attention_do_gb300" / "csrc" / "k_tc_dkdv.cu")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_source_hash("dkdv_tc")
    entry = {"dkdv_tc": {"source_sha": sha, "bytes_per_launch_full": 1234}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(entry))
    assert bench.traffic_for("dkdv_tc") == 1234
    assert bench.traffic_for("dq_tc") is None  # no entry
    # the kernel changed since the capture: no figure
    with open(tmp_path / "block_sparse_attention_do_gb300" / "csrc" / "k_tc_dkdv.cu", "a") as f:
        f.write("// changed\n")
    assert bench.traffic_for("dkdv_tc") is None
