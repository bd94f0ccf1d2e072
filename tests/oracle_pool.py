"""The CPU oracle over a pool of worker processes, for full-size parity checks.

The oracle's weighted sum over experts is linear in the set of experts it
visits, so the routed experts are split into chunks, each worker runs the oracle
on the slots routed to its chunk (the other slots are masked out, which the
oracle skips) for the requested tokens, and the partial outputs are added. Each
worker regenerates the seeded inputs and only the expert weights it needs. The
pool is created with the "spawn" start method, so it is safe after CUDA has been
initialised in the parent."""
import multiprocessing as mp
import os

import numpy as np

import oracle
from int4_weight_only_moe_gb300 import inputs


def _routed(wl, step):
    hidden, logits = inputs.workload_inputs(wl, step=step)
    ids, w = oracle.route(logits, wl.topk)
    return hidden, ids, w.astype(np.float32)


def _partial(task):
    fields, step, experts, tokens = task
    wl = inputs.Workload(*fields)
    hidden, ids, w = _routed(wl, step)
    masked = np.where(np.isin(ids, experts), ids, -1).astype(np.int32)
    return oracle.moe_forward(hidden, masked, w, None, None, None, None, tokens=tokens,
                              expert_source=lambda e: inputs.expert_weights(e, wl.K, wl.N))


def workload_fields(wl):
    return (wl.name, wl.E, wl.K, wl.N, wl.topk, wl.M, wl.routing, wl.zipf_s)


def oracle_rows(wl, tokens, step=0, procs=None):
    """Oracle output rows ``tokens`` of workload ``wl`` (float64 [len(tokens), K])."""
    _, ids, _ = _routed(wl, step)
    tokens = np.asarray(tokens)
    experts = np.unique(ids[tokens])
    procs = procs or max(1, min(os.cpu_count() or 1, 32))
    chunks = [c for c in np.array_split(experts, min(len(experts), 4 * procs)) if len(c)]
    tasks = [(workload_fields(wl), step, c, tokens) for c in chunks]
    env = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in env:
        os.environ[k] = "1"  # one BLAS thread per worker
    try:
        with mp.get_context("spawn").Pool(min(procs, len(tasks))) as pool:
            parts = pool.map(_partial, tasks)
    finally:
        for k, v in env.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return np.sum(parts, axis=0)
