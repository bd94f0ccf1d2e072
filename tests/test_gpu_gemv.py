"""The small-batch CUDA-core path (by default up to 256 routed slots: tiles of at
most 4 token rows per expert, both products as matrix-vector products) against
the oracle and against the tensor-core kernels on the same inputs, through the
C-ABI.

Covered: every grid size from one CTA (every unit in one CTA's sequence) to more
CTAs than steps; experts with 1..16 rows (several 4-row tiles of one expert);
batches up to 32 slots (routed inside the kernels) and above (the align kernel's
tile list); skipped ids; a batch with no valid slot; the give-up path of every
small-batch path; both products in one launch against two; every output element
written; and the intermediate activations. The two paths compute the same products from
differently rounded activations (the tensor cores read them as fp16, the CUDA
cores as 16-bit block fixed point per scale group), so the intermediate may
differ by about one fp16 unit and the output accumulators by about 2^-12 of
their magnitude (the oracle comparison is the parity check proper)."""
import numpy as np
import pytest
import torch

import int4_weight_only_moe_gb300 as pkg
import oracle
from int4_weight_only_moe_gb300 import inputs
from tests.gpu_helpers import (Problem, assert_close, bf16_tensor_to_f64, bits16, check_accumulator, dev,
                               workload_inputs)

pytestmark = pytest.mark.gpu
GEMV_DEFAULT = 1  # the CUDA-core path for batches of at most 256 routed slots


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def run_path(prob, hidden, ids, wts, gemv, one_launch=0):
    pkg.moe_w4a16_set_option(prob.moe.handle, pkg.OPT_GEMV_SMALL_BATCH, gemv)
    pkg.moe_w4a16_set_option(prob.moe.handle, pkg.OPT_GEMV_ONE_LAUNCH, one_launch)
    try:
        got = prob.run(hidden, ids, wts)
        status = prob.moe.status()
        M = hidden.shape[0]
        acc = prob.moe.accumulator(M).cpu().numpy().astype(np.float64)
        inter = prob.moe.intermediate(M).cpu().numpy().astype(np.float64)
        bits = inputs.f32_to_bf16_bits(got.astype(np.float32))  # (exact: got holds bf16 values)
    finally:
        pkg.moe_w4a16_set_option(prob.moe.handle, pkg.OPT_GEMV_SMALL_BATCH, GEMV_DEFAULT)
        pkg.moe_w4a16_set_option(prob.moe.handle, pkg.OPT_GEMV_ONE_LAUNCH, 0)
    return got, status, acc, inter, bits


def compare_paths(prob, hidden, ids, wts, what, ref_ids=None, gemv=1):
    ref = prob.reference(hidden, ids if ref_ids is None else ref_ids, wts)
    g_out, g_st, g_acc, g_h, g_bits = run_path(prob, hidden, ids, wts, gemv=gemv)
    t_out, t_st, t_acc, t_h, _ = run_path(prob, hidden, ids, wts, gemv=0)
    assert g_st == t_st, (g_st, t_st)
    if np.any(ref != 0):
        assert_close(g_out, ref, f"{what} (CUDA cores)")
        assert_close(t_out, ref, f"{what} (tensor cores)")
        check_accumulator(g_acc, g_bits, ref, f"{what} (CUDA cores)")
    else:
        assert np.all(g_out == 0) and np.all(t_out == 0)
    scale = float(np.abs(t_acc).max()) or 1.0
    np.testing.assert_allclose(g_acc, t_acc, rtol=2.0 ** -9, atol=2.0 ** -10 * scale, err_msg=what)
    hs = float(np.abs(t_h).max()) or 1.0
    np.testing.assert_allclose(g_h, t_h, rtol=2.0 ** -9, atol=2.0 ** -12 * hs, err_msg=what + " intermediate")
    return g_st


@pytest.mark.parametrize("num_ctas", [None, 1, 3, 7, 64, 256])
@pytest.mark.parametrize("M", [1, 2, 3, 8])
def test_gemv_matches_oracle_and_tensor_cores(M, num_ctas):
    # E=16, K=512, N=256, top-4: 4 steps per gate/up unit, 2 per down unit; 3 and 7
    # CTAs cut units between CTAs at odd places, 256 leaves most CTAs no step
    E, K, N, k = 16, 512, 256, 4
    prob = Problem(E, K, N, k, num_ctas=num_ctas)
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    hidden, ids, wts = workload_inputs(wl, step=M)
    assert compare_paths(prob, hidden, ids, wts, f"M={M} ctas={num_ctas}") == 0
    prob.close()


def test_gemv_option_values():
    # 1 (default) and 3: batches of up to 256 slots; 2: single-token batches only;
    # 0: never; anything else is rejected
    prob = Problem(8, 256, 128, 2)
    h = prob.moe.handle
    for v in (0, 1, 2, 3):
        pkg.moe_w4a16_set_option(h, pkg.OPT_GEMV_SMALL_BATCH, v)
    with pytest.raises(pkg.MoeW4A16Error):
        pkg.moe_w4a16_set_option(h, pkg.OPT_GEMV_SMALL_BATCH, 4)
    prob.close()


@pytest.mark.parametrize("num_ctas", [None, 1, 5, 256])
@pytest.mark.parametrize("M", [9, 37, 64])
def test_gemv_align_tile_list(M, num_ctas):
    # more than 32 routed slots (up to 256): the align kernel writes
    # the tile list and the CUDA-core kernels read it (1 CTA: every tile through
    # the global-memory fallback of the kernel's tile window)
    E, K, N, k = 16, 512, 256, 4
    prob = Problem(E, K, N, k, num_ctas=num_ctas)
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    hidden, ids, wts = workload_inputs(wl, step=M)
    assert compare_paths(prob, hidden, ids, wts, f"tile list M={M} ctas={num_ctas}", gemv=3) == 0
    prob.close()


@pytest.mark.parametrize("rows", [4, 5, 9, 16])
def test_gemv_expert_with_many_rows(rows):
    # one expert receives `rows` of the batch's slots: ceil(rows / 4) tiles of it,
    # each streaming the expert's weights (topk 2, 16 tokens: 32 slots)
    E, K, N, k, M = 8, 768, 384, 2, 16
    prob = Problem(E, K, N, k, num_ctas=5)
    rng = np.random.default_rng(rows)
    ids = np.zeros((M, k), dtype=np.int32)
    for t in range(M):
        ids[t] = rng.choice(np.arange(1, E), size=k, replace=False)
    ids[:rows, 0] = 0  # expert 0 (never drawn above) in `rows` tokens' first slot
    hidden = inputs.hidden_states(M, K)
    wts = rng.uniform(0.1, 1.0, size=(M, k)).astype(np.float32)
    compare_paths(prob, hidden, ids, wts, f"{rows} rows on one expert")
    prob.close()


def test_gemv_skipped_ids_and_empty_batch():
    E, K, N, k, M = 8, 512, 256, 4, 3
    prob = Problem(E, K, N, k)
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    hidden, ids, wts = workload_inputs(wl)
    bad = ids.copy()
    bad[0, 1] = E + 3
    bad[2, 3] = -1
    st = compare_paths(prob, hidden, bad, wts, "skipped ids", ref_ids=np.where(bad >= E, -1, bad))
    assert st == pkg.STATUS_BAD_EXPERT_ID
    none = np.full_like(ids, E + 1)
    st = compare_paths(prob, hidden, none, wts, "no valid slot", ref_ids=np.full_like(ids, -1))
    assert st == pkg.STATUS_BAD_EXPERT_ID
    prob.close()


def test_gemv_intermediate_matches_oracle():
    # h = SiLU(gate) * up of every routed row, element by element
    E, K, N, k, M = 8, 1024, 512, 4, 2
    prob = Problem(E, K, N, k, num_ctas=11)
    pkg.moe_w4a16_set_option(prob.moe.handle, pkg.OPT_GEMV_SMALL_BATCH, 1)
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    hidden, ids, wts = workload_inputs(wl)
    prob.run(hidden, ids, wts)
    assert prob.moe.status() == 0
    h_rows = bf16_tensor_to_f64(prob.moe.intermediate(M))
    x = oracle.bf16_to_f64(hidden)
    ref = np.zeros_like(h_rows)
    for t in range(M):
        for j in range(k):
            w1, _ = oracle.expert_dense(*prob.w, int(ids[t, j]))
            ref[t * k + j] = oracle.expert_hidden(x[t:t + 1], w1)[0]
    assert_close(h_rows, ref, "intermediate (CUDA cores)", bf16_output=False)
    prob.close()


def test_both_small_batch_paths_give_up_cleanly():
    # the give-up hook on each small-batch path in turn (CUDA cores in one launch,
    # in two, tensor cores); the next call is clean
    E, K, N, k, M = 8, 512, 256, 4, 2
    prob = Problem(E, K, N, k)
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    hidden, ids, wts = workload_inputs(wl)
    h = prob.moe.handle
    for gemv, one in ((1, 1), (1, 0), (0, 1)):
        pkg.moe_w4a16_set_option(h, pkg.OPT_GEMV_SMALL_BATCH, gemv)
        pkg.moe_w4a16_set_option(h, pkg.OPT_GEMV_ONE_LAUNCH, one)
        pkg.moe_w4a16_set_option(h, pkg.OPT_WAIT_LIMIT_US, 1000)
        pkg.moe_w4a16_set_option(h, pkg.OPT_TEST_WAIT_NEVER_COMPLETES, 1)
        prob.run(hidden, ids, wts)
        assert prob.moe.status() & pkg.STATUS_TIMEOUT
        pkg.moe_w4a16_set_option(h, pkg.OPT_TEST_WAIT_NEVER_COMPLETES, 0)
        pkg.moe_w4a16_set_option(h, pkg.OPT_WAIT_LIMIT_US, 0)
        got = prob.run(hidden, ids, wts)
        assert prob.moe.status() == 0
        assert_close(got, prob.reference(hidden, ids, wts), f"after give-up, gemv={gemv} one launch={one}")
    pkg.moe_w4a16_set_option(h, pkg.OPT_GEMV_SMALL_BATCH, GEMV_DEFAULT)
    pkg.moe_w4a16_set_option(h, pkg.OPT_GEMV_ONE_LAUNCH, 0)
    prob.close()


@pytest.mark.parametrize("num_ctas", [None, 1, 3, 7, 64])
@pytest.mark.parametrize("M", [1, 2, 3, 8])
def test_gemv_one_launch_matches_two_launches(M, num_ctas):
    # both products in one cooperative launch (at most 32 slots): the same
    # arithmetic as the two launches, so the intermediate is identical bit for bit
    # (the split units' sums run in CTA order either way); the output differs
    # only by the order of the fp32 atomic adds, and both match the oracle.
    # 1 CTA: every step row of the intermediate comes from the CTA itself; 7 and
    # 64 CTAs cut the products' units at different places
    E, K, N, k = 16, 512, 256, 4
    prob = Problem(E, K, N, k, num_ctas=num_ctas)
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    hidden, ids, wts = workload_inputs(wl, step=M + 7)
    ref = prob.reference(hidden, ids, wts)
    o_out, o_st, o_acc, o_h, o_bits = run_path(prob, hidden, ids, wts, gemv=1, one_launch=1)
    t_out, t_st, t_acc, t_h, _ = run_path(prob, hidden, ids, wts, gemv=1, one_launch=0)
    assert o_st == 0 and t_st == 0
    np.testing.assert_array_equal(o_h, t_h)
    assert_close(o_out, ref, f"one launch M={M} ctas={num_ctas}")
    check_accumulator(o_acc, o_bits, ref, f"one launch M={M} ctas={num_ctas}")
    scale = float(np.abs(t_acc).max()) or 1.0
    np.testing.assert_allclose(o_acc, t_acc, rtol=2.0 ** -16, atol=2.0 ** -18 * scale)
    prob.close()


@pytest.mark.parametrize("case", ["routed", "no valid slot"])
@pytest.mark.parametrize("num_ctas", [None, 1, 7])
def test_gemv_writes_every_output_element(case, num_ctas):
    # an output buffer filled with NaNs beforehand comes back fully written, equal
    # to the rounding of the accumulator, with tokens that have no valid slot (and
    # a batch with none at all) as zeros
    E, K, N, k, M = 8, 512, 256, 4, 5
    prob = Problem(E, K, N, k, num_ctas=num_ctas)
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    hidden, ids, wts = workload_inputs(wl)
    ids = ids.copy()
    if case == "routed":
        ids[2, :] = E + 1  # token 2: no valid slot
    else:
        ids[:] = -1
    out = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    prob.moe.forward(dev(bits16(hidden)), dev(ids), dev(wts), out=out)
    torch.cuda.synchronize()
    got = bf16_tensor_to_f64(out)
    assert np.all(np.isfinite(got))
    acc = prob.moe.accumulator(M).cpu().numpy()
    np.testing.assert_array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16),
                                  inputs.f32_to_bf16_bits(acc.astype(np.float32)))
    ref = prob.reference(hidden, np.where((ids < 0) | (ids >= E), -1, ids), wts)
    if case == "routed":
        assert np.all(got[2] == 0)
        assert_close(got, ref, "every element written")
    else:
        assert np.all(got == 0)
    prob.close()
