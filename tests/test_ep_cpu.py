"""Expert parallelism on the host (gloo, world size 2 and 3): the expert
partition, the per-rank partial sums and the one sum-reduce that combines them.
The ranks' partials are the oracle's forward restricted to each rank's experts
(slots routed elsewhere are skipped, exactly as the library's expert-range
handles do); their all-reduced sum must equal the full oracle forward."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from int4_weight_only_moe_gb300 import ep, inputs


def test_expert_range_partitions_the_layer():
    for E in (1, 2, 7, 16, 384):
        for world in range(1, min(E, 9) + 1):
            ranges = [ep.expert_range(E, world, r) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == E
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
            sizes = [e - b for b, e in ranges]
            assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        ep.expert_range(2, 3, 0)
    with pytest.raises(ValueError):
        ep.expert_range(8, 2, 2)


def local_ids(ids, begin, end):
    """The layer's ids as indices into experts [begin, end); slots routed to other
    experts become -1 (skipped by the oracle)."""
    return np.where((ids >= begin) & (ids < end), ids - begin, -1).astype(np.int32)


PROBLEM = dict(E=7, K=64, N=32, M=6, k=3)


def problem():
    import oracle
    p = PROBLEM
    ws = [inputs.expert_weights(e, p["K"], p["N"]) for e in range(p["E"])]
    w = [np.stack([x[i] for x in ws]) for i in range(4)]
    hidden, logits = inputs.workload_inputs(inputs.Workload("ep", p["E"], p["K"], p["N"], p["k"],
                                                            p["M"], "normal"))
    ids, wts = oracle.route(logits, p["k"])
    return w, hidden, ids, wts


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, hidden, ids, wts = problem()
    b, e = ep.expert_range(PROBLEM["E"], world, rank)
    # this rank's experts only: the handle holds weights [b, e) and sees local ids
    part = oracle.moe_forward(hidden, local_ids(ids, b, e), wts, *(a[b:e] for a in w))
    t = torch.from_numpy(part.copy())
    ep.allreduce_partial(t)
    q.put((rank, (b, e), t.numpy()))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_allreduced_partials_equal_the_full_layer(world):
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=120) for _ in procs), key=lambda g: g[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w, hidden, ids, wts = problem()
    full = oracle.moe_forward(hidden, ids, wts, *w)
    for rank, rng, summed in got:
        assert rng == ep.expert_range(PROBLEM["E"], world, rank)
        np.testing.assert_allclose(summed, full, rtol=1e-12, atol=1e-12)
    # and no single rank's partial is the whole (each rank holds part of the routing)
    b, e = ep.expert_range(PROBLEM["E"], world, 0)
    only0 = oracle.moe_forward(hidden, local_ids(ids, b, e), wts, *(a[b:e] for a in w))
    assert not np.allclose(only0, full)
