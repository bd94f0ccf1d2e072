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


class _FakePool:
    procs = 4

    def __init__(self, *a, **k):
        pass

    def close(self):
        pass


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    called = []
    monkeypatch.setattr(bench, "OraclePool", _FakePool)
    monkeypatch.setattr(bench, "oracle_call", lambda pool, wl, s: called.append(s) or (0.1, 8))
    bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3"])
    assert called == [] and capsys.readouterr().out == ""


def test_reference_arm_line(monkeypatch, capsys):
    # the reference arm honours --steps and --warmup and reports the GPU arm's config
    import json
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    called = []
    monkeypatch.setattr(bench, "OraclePool", _FakePool)
    monkeypatch.setattr(bench, "oracle_call", lambda pool, wl, s: called.append(s) or (0.5, 8))
    bench.main(["--impl", "reference", "--steps", "4", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip())
    assert called == list(range(7))
    assert line["impl"] == "reference" and line["value"] == pytest.approx(2.0)
    assert line["steps"] == 4 and line["warmup"] == 3
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["config"] == bench.headline_config(bench.inputs.WORKLOADS["decode"], 1)
    assert line["cpu_baseline"]["cores"] == 4


def test_oracle_pool_times_expert_shares():
    # the pooled oracle timing runs real oracle arithmetic on a tiny workload
    import bench
    wl = bench.inputs.WORKLOADS["tiny"]
    pool = bench.OraclePool(procs=2)
    try:
        wall, n = bench.oracle_call(pool, wl, 0)
    finally:
        pool.close()
    assert n >= 1 and wall > 0
