"""The multi-process path of bench.py on CPU (gloo, world size 2): independent
replicas whose timed region is reduced with a max over ranks, and a reference
arm that only rank 0 runs."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    slowest = bench.reduce_max(10.0 * (rank + 1), torch.device("cpu"))
    dist.barrier()
    q.put((rank, slowest, bench.dist_env()))
    dist.destroy_process_group()


def test_replica_time_is_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [20.0, 20.0]
    assert [g[2] for g in got] == [(0, 0, 2), (1, 1, 2)]


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    called = []
    monkeypatch.setattr(bench, "oracle_step", lambda wl, s: called.append(s) or 0.1)
    bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3"])
    assert called == [] and capsys.readouterr().out == ""


def test_reference_arm_line(monkeypatch, capsys):
    import json
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setattr(bench, "oracle_step", lambda wl, s: 0.5)
    bench.main(["--impl", "reference", "--steps", "4", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["value"] == pytest.approx(2.0)
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
