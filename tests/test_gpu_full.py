"""Full-size parity: E=384 experts, hidden 7168, intermediate 2048, top-8, INT4
group 32 (the MoE layer the pages benchmark), every batch size of the sweep, in
the launch configuration the benchmark times (persistent grid of one CTA per SM,
programmatic dependent launch).

Every output row is compared with the oracle up to M = 90 tokens (the oracle runs
expert by expert over a pool of host processes); the larger batches are compared
on 64 sampled tokens plus every token in the last (ragged) token tile of the
hottest expert, where a tile-boundary mistake would sit. The margins to the
tolerance (relative L2 error, largest error over the reference RMS) of every
configuration are printed in the session summary. Also here, because they need
the full-size weights: the intermediate activations of a decode step, and the
cost-weighted stream-K boundaries at M = 1024 against a brute-force enumeration."""
import numpy as np
import pytest
import torch

import int4_weight_only_moe_gb300 as pkg
import oracle
from int4_weight_only_moe_gb300 import inputs
from tests import oracle_pool
from tests.conftest import MARGINS
from tests.gpu_helpers import (TOL_MAX_OVER_RMS, TOL_REL_L2, Problem, assert_close, bf16_tensor_to_f64,
                               bits16, check_accumulator, dev, errors, excess_over_rounding,
                               workload_inputs)

pytestmark = pytest.mark.gpu

ALL_ROWS = ["decode", "small9", "small32", "small90"]
SAMPLED = ["plateau256", "plateau512", "large_uniform", "large_zipf"]
TILE = 64  # largest token tile (rows) of the GEMMs


@pytest.fixture(scope="module")
def full_problem():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    wl = inputs.WORKLOADS["decode"]
    prob = Problem(wl.E, wl.K, wl.N, wl.topk)
    yield prob
    prob.close()


def hottest_last_tile_tokens(ids, E):
    """Tokens of the rows in the last token tile of the expert with the most rows."""
    sorted_ids, offsets, _ = oracle.moe_align(ids, E, 16)
    counts = np.bincount(ids.reshape(-1), minlength=E)
    hot = int(counts.argmax())
    seg = sorted_ids[offsets[hot]:offsets[hot + 1]]
    last = seg[(len(seg) - 1) // TILE * TILE:]
    real = last[last < ids.size]
    return np.unique(real // ids.shape[1])


def sample_tokens(ids, E, n, rng):
    M = ids.shape[0]
    picks = set(rng.choice(M, size=min(n, M), replace=False).tolist()) | {0, M - 1}
    picks |= set(hottest_last_tile_tokens(ids, E).tolist())
    return np.array(sorted(picks))


def record(name, toks, got, ref, acc=None):
    rel, mx = errors(got, ref)
    line = (f"{name}: {len(toks)} tokens, bf16 out rel L2 {rel:.3e} (limit {TOL_REL_L2:g}), "
            f"max|d|/rms {mx:.3e}, beyond bf16 rounding {excess_over_rounding(got, ref):.3e} "
            f"(limit {TOL_MAX_OVER_RMS:g})")
    if acc is not None:
        arel, amx = errors(acc, ref)
        line += f"; fp32 accumulator rel L2 {arel:.3e}, max|d|/rms {amx:.3e}"
    MARGINS.append(line)


def run_with_accumulator(prob, hidden, ids, wts):
    out = prob.moe.forward(dev(bits16(hidden)), dev(ids), dev(wts))
    torch.cuda.synchronize()
    acc = prob.moe.accumulator(hidden.shape[0]).cpu().numpy().astype(np.float64)
    return bf16_tensor_to_f64(out), out.view(torch.int16).cpu().numpy(), acc


@pytest.mark.parametrize("name", ALL_ROWS + SAMPLED)
def test_full_size_parity(full_problem, name):
    wl = inputs.WORKLOADS[name]
    hidden, ids, wts = workload_inputs(wl)
    got, bits, acc = run_with_accumulator(full_problem, hidden, ids, wts)
    assert np.all(np.isfinite(got))
    assert full_problem.moe.status() == 0
    if name in ALL_ROWS:
        toks = np.arange(wl.M)
    else:
        toks = sample_tokens(ids, wl.E, 64, np.random.default_rng(len(name)))
    ref = oracle_pool.oracle_rows(wl, toks)
    record(name, toks, got[toks], ref, acc[toks])
    assert_close(got[toks], ref, f"{name} ({len(toks)} tokens)")
    check_accumulator(acc[toks], bits[toks], ref, name)
    # every output element is the exact rounding of its accumulator
    np.testing.assert_array_equal(bits.view(np.uint16), inputs.f32_to_bf16_bits(acc.astype(np.float32)))


def test_full_size_zipf_small_batch_cuda_cores(full_problem):
    # 32 Zipf-routed tokens (256 routed slots) run on the CUDA cores by default:
    # the hottest experts take several 4-row tiles, and tiles of 1..4 rows mix
    # under the cost-weighted split; every row against the oracle
    wl = inputs.Workload("small32_zipf", 384, 7168, 2048, 8, 32, "zipf")
    hidden, ids, wts = workload_inputs(wl)
    counts = np.bincount(ids.reshape(-1), minlength=wl.E)
    assert counts.max() > 4 and np.any((counts > 1) & (counts < 4))  # several tiles; mixed tile sizes
    got, bits, acc = run_with_accumulator(full_problem, hidden, ids, wts)
    assert full_problem.moe.status() == 0
    toks = np.arange(wl.M)
    ref = oracle_pool.oracle_rows(wl, toks)
    record("small32 Zipf (CUDA cores, multi-tile experts)", toks, got, ref, acc)
    assert_close(got, ref, "small32 Zipf")
    check_accumulator(acc, bits, ref, "small32 Zipf")
    np.testing.assert_array_equal(bits.view(np.uint16), inputs.f32_to_bf16_bits(acc.astype(np.float32)))


def test_decode_intermediate_full_size(full_problem):
    # SiLU(gate) * up of the 8 routed rows of a decode step, element by element
    wl = inputs.WORKLOADS["decode"]
    hidden, ids, wts = workload_inputs(wl, step=3)
    full_problem.run(hidden, ids, wts)
    h_rows = bf16_tensor_to_f64(full_problem.moe.intermediate(wl.M))
    x = oracle.bf16_to_f64(hidden)
    ref = np.zeros_like(h_rows)
    for j in range(wl.topk):
        q1, s1, _, _ = inputs.expert_weights(int(ids[0, j]), wl.K, wl.N)
        ref[j] = oracle.expert_hidden(x[:1], oracle.dequantize(q1, s1))[0]
    record("decode intermediate h (fp16 operand)", np.arange(wl.topk), h_rows, ref)
    assert_close(h_rows, ref, "decode intermediate", bf16_output=False)


def enumerate_boundaries(ids, E, R, KB, G, per_group):
    """First step of every CTA's share, by enumeration: every step of every unit
    (expert, row tile, token tile) in order with its cost 8 + c * max(0, groups - 2);
    CTA c starts at the first step whose preceding cost reaches floor(c * total / G)."""
    _, offsets, _ = oracle.moe_align(ids, E, 16)
    pads = np.diff(offsets.astype(np.int64))
    unit_costs = []
    for e in range(E):
        tiles = [min(TILE, int(pads[e]) - t * TILE) // 16 for t in range(-(-int(pads[e]) // TILE))]
        costs = [8 + per_group * max(0, g - 2) for g in tiles]
        for _ in range(R):
            unit_costs.extend(costs)
    steps = np.repeat(np.array(unit_costs, dtype=np.int64), KB)
    before = np.concatenate([[0], np.cumsum(steps)])
    total = int(before[-1])
    starts = [int(np.searchsorted(before, (c * total) // G, side="left")) for c in range(G)]
    return starts + [len(steps)], before


def test_stream_k_boundaries_match_enumeration(full_problem):
    wl = inputs.WORKLOADS["large_zipf"]
    hidden, ids, wts = workload_inputs(wl)
    h = full_problem.moe.handle
    pkg.moe_w4a16_set_option(h, pkg.OPT_STEP_COST_GATEUP, 3)
    pkg.moe_w4a16_set_option(h, pkg.OPT_STEP_COST_DOWN, 2)
    try:
        got, bits, acc = run_with_accumulator(full_problem, hidden, ids, wts)
        G = torch.cuda.get_device_properties(0).multi_processor_count
        bounds, flags = pkg.moe_w4a16_schedule_debug(h, full_problem.moe.workspace, wl.M, min(G, 256))
    finally:
        pkg.moe_w4a16_set_option(h, pkg.OPT_STEP_COST_GATEUP, 0)
        pkg.moe_w4a16_set_option(h, pkg.OPT_STEP_COST_DOWN, 2)
    assert full_problem.moe.status() == 0
    assert flags == 3
    G = len(bounds[0]) - 1
    for w, (R, KB, c) in enumerate([(2 * wl.N // 128, wl.K // 128, 3), (wl.K // 128, wl.N // 128, 2)]):
        want, before = enumerate_boundaries(ids, wl.E, R, KB, G, c)
        assert bounds[w] == want, f"GEMM {w}"
        # every share carries the average cost to within one step's cost
        share = np.diff(before[np.array(want)])
        assert share.max() <= before[-1] / G + 8 + 2 * c
    toks = sample_tokens(ids, wl.E, 16, np.random.default_rng(5))
    ref = oracle_pool.oracle_rows(wl, toks)
    record("large_zipf, both GEMMs cost-weighted", toks, got[toks], ref, acc[toks])
    assert_close(got[toks], ref, "weighted split, both GEMMs")
    check_accumulator(acc[toks], bits[toks], ref, "weighted split, both GEMMs")
