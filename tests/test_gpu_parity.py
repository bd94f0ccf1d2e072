"""CUDA path vs the CPU oracle on seeded inputs, through the C-ABI (small and
medium shapes that still span several tiles, ragged tails and split units).

Bit-exact: the align (sorted ids, offsets, padded length) and the repack round
trip. Floating point: relative L2 error <= 5e-3 and max |error| <= 2e-2 * rms of
the reference, for the output and for the intermediate activations."""
import numpy as np
import pytest
import torch

import int4_weight_only_moe_gb300 as pkg
import oracle
from int4_weight_only_moe_gb300 import inputs
from tests.gpu_helpers import Problem, assert_close, bf16_tensor_to_f64, bits16, dev, workload_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def zipf_ids(rng, M, E, k, s=1.1):
    p = np.arange(1, E + 1, dtype=float) ** -s
    p /= p.sum()
    perm = rng.permutation(E)
    return np.stack([perm[rng.choice(E, size=k, replace=False, p=p)] for _ in range(M)]).astype(np.int32)


# ---------------------------------------------------------------------------- align


@pytest.mark.parametrize("M,k,E,block,dist", [
    (0, 8, 16, 16, "uniform"), (1, 8, 384, 16, "uniform"), (4, 2, 8, 16, "uniform"),
    (9, 8, 384, 16, "uniform"), (90, 8, 384, 16, "uniform"), (1024, 8, 384, 16, "uniform"),
    (1024, 8, 384, 16, "zipf"), (333, 3, 1024, 64, "uniform"), (77, 5, 40, 1, "zipf"),
    (500, 4, 7, 5, "dup"), (4096, 8, 384, 16, "zipf"),
    # at most 32 slots: the one-warp path
    (3, 8, 384, 16, "dup"), (2, 8, 40, 5, "zipf"), (4, 8, 384, 1, "uniform"), (1, 4, 3, 64, "dup"),
    (16, 2, 1024, 16, "uniform"), (5, 6, 12, 16, "dup"),
])
def test_align_bit_exact(M, k, E, block, dist):
    rng = np.random.default_rng(M * 31 + E)
    if dist == "uniform":
        ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(M)]).astype(np.int32) \
            if M else np.zeros((0, k), np.int32)
    elif dist == "zipf":
        ids = zipf_ids(rng, M, E, k)
    else:  # duplicates inside a token are still well defined
        ids = rng.integers(0, E, size=(M, k)).astype(np.int32)
    ref_sorted, ref_off, ref_n = oracle.moe_align(ids, E, block)
    MK = M * k
    cap = MK + min(E, MK) * (block - 1) + 1
    d_ids = dev(ids) if M else torch.zeros(1, dtype=torch.int32, device="cuda")
    d_sorted = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
    d_off = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    d_n = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkg.moe_w4a16_align_debug(d_ids, M, k, E, block, d_sorted, d_off, d_n)
    torch.cuda.synchronize()
    n = int(d_n.item())
    assert n == ref_n
    np.testing.assert_array_equal(d_sorted.cpu().numpy()[:n], ref_sorted)
    np.testing.assert_array_equal(d_off.cpu().numpy(), ref_off)


def test_align_small_batch_skips_out_of_range_ids():
    # the one-warp path (at most 32 slots) flags and skips bad ids like the general one
    ids = np.array([[3, 3, -1, 7], [12, 0, 3, 1 << 30], [5, 5, 5, 11]], dtype=np.int32)
    ref_sorted, ref_off, ref_n = oracle.moe_align(ids, 12, 16)
    cap = 12 + 12 * 15
    d_sorted = torch.zeros(cap, dtype=torch.int32, device="cuda")
    d_off = torch.zeros(13, dtype=torch.int32, device="cuda")
    d_n = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkg.moe_w4a16_align_debug(dev(ids), 3, 4, 12, 16, d_sorted, d_off, d_n)
    torch.cuda.synchronize()
    n = int(d_n.item())
    assert n == ref_n
    np.testing.assert_array_equal(d_sorted.cpu().numpy()[:n], ref_sorted)
    np.testing.assert_array_equal(d_off.cpu().numpy(), ref_off)


def test_align_skips_out_of_range_ids():
    rng = np.random.default_rng(0)
    ids = rng.integers(0, 12, size=(50, 4)).astype(np.int32)
    ids[3, 2] = -1
    ids[10, 0] = 12
    ids[11, 1] = 1 << 30
    ref_sorted, ref_off, ref_n = oracle.moe_align(ids, 12, 16)
    cap = 50 * 4 + 12 * 15
    d_sorted = torch.zeros(cap, dtype=torch.int32, device="cuda")
    d_off = torch.zeros(13, dtype=torch.int32, device="cuda")
    d_n = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkg.moe_w4a16_align_debug(dev(ids), 50, 4, 12, 16, d_sorted, d_off, d_n)
    torch.cuda.synchronize()
    n = int(d_n.item())
    assert n == ref_n
    np.testing.assert_array_equal(d_sorted.cpu().numpy()[:n], ref_sorted)


# ---------------------------------------------------------------------------- repack


@pytest.mark.parametrize("E,K,N", [(8, 256, 128), (3, 1024, 512), (2, 7168, 2048)])
def test_pack_roundtrip_bit_exact(E, K, N):
    w1_q, w1_s, w2_q, w2_s = inputs.all_expert_weights(E, K, N, seed=5)
    moe = pkg.MoEW4A16(E, K, N, 2)
    moe.pack(dev(w1_q), dev(bits16(w1_s)), dev(w2_q), dev(bits16(w2_s)))
    assert pkg.moe_w4a16_packed_bytes(moe.handle) == E * oracle.roofline_bytes_per_expert(K, N)
    outs = [torch.zeros_like(dev(a)) for a in (w1_q, bits16(w1_s), w2_q, bits16(w2_s))]
    pkg.moe_w4a16_unpack_debug(moe.handle, *outs)
    torch.cuda.synchronize()
    for got, ref in zip(outs, (w1_q, bits16(w1_s), w2_q, bits16(w2_s))):
        np.testing.assert_array_equal(got.cpu().numpy(), ref)
    moe.close()


# ---------------------------------------------------------------------------- forward


def assert_within_one_ulp(a, b):
    """Two bf16 results of the same kernels equal up to one unit in the last place of
    the larger one, plus the fp32 summation-order term.

    The down projection's partial sums reach the fp32 accumulator through atomic
    adds whose order varies between calls. Two orders of the same T terms differ by
    at most 2(T-1)u times the sum of the terms' magnitudes (u = 2^-24); near zero this
    exceeds the bf16 unit, so an absolute floor of 2^-16 times the output's largest
    magnitude (room for T * sum|terms| up to 128 times that magnitude) is allowed.
    """
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(a), np.abs(b)) + 1e-30)) - 7)
    floor = np.exp2(-16.0) * max(float(np.abs(b).max()), 1e-30)
    assert np.all(np.abs(a - b) <= ulp + floor)


def check_forward(prob, hidden, ids, wts, what):
    got = prob.run(hidden, ids, wts)
    ref = prob.reference(hidden, ids, wts)
    assert_close(got, ref, what)
    assert prob.moe.status() == 0
    return got


def test_tiny_forward_and_intermediate():
    wl = inputs.WORKLOADS["tiny"]
    prob = Problem(wl.E, wl.K, wl.N, wl.topk)
    hidden, ids, wts = workload_inputs(wl)
    check_forward(prob, hidden, ids, wts, "tiny")
    h_rows = bf16_tensor_to_f64(prob.moe.intermediate(wl.M))
    x = oracle.bf16_to_f64(hidden)
    ref_h = np.zeros_like(h_rows)
    for t in range(wl.M):
        for j in range(wl.topk):
            w1, _ = oracle.expert_dense(*prob.w, int(ids[t, j]))
            ref_h[t * wl.topk + j] = oracle.expert_hidden(x[t:t + 1], w1)[0]
    assert_close(h_rows, ref_h, "tiny intermediate", bf16_output=False)
    prob.close()


@pytest.mark.parametrize("num_ctas", [None, 1, 3, 64, 256])
@pytest.mark.parametrize("M", [1, 5, 37, 200])
def test_mid_forward_grid_sizes(M, num_ctas):
    E, K, N, k = 16, 512, 256, 4
    prob = Problem(E, K, N, k, num_ctas=num_ctas)
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    hidden, ids, wts = workload_inputs(wl)
    check_forward(prob, hidden, ids, wts, f"mid M={M} ctas={num_ctas}")
    prob.close()


@pytest.mark.parametrize("num_ctas", [None, 1, 3, 64])
@pytest.mark.parametrize("M", [1, 2, 8])
def test_fused_small_batch_matches_two_launches(M, num_ctas):
    # at most 32 routed slots: both GEMMs in one cooperative launch (the down
    # phase waits per token tile for the intermediate) against the two-launch path
    # and the oracle; 1 and 3 CTAs put many gate/up and down units in one CTA's
    # sequence, 64 leaves some CTAs a share of only a few steps
    E, K, N, k = 16, 512, 256, 4
    prob = Problem(E, K, N, k, num_ctas=num_ctas)
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    hidden, ids, wts = workload_inputs(wl, step=M)
    pkg.moe_w4a16_set_option(prob.moe.handle, pkg.OPT_FUSED_SMALL_BATCH, 1)
    fused = check_forward(prob, hidden, ids, wts, f"fused M={M} ctas={num_ctas}")
    pkg.moe_w4a16_set_option(prob.moe.handle, pkg.OPT_FUSED_SMALL_BATCH, 0)
    # (against the two tensor-core launches: the same arithmetic)
    pkg.moe_w4a16_set_option(prob.moe.handle, pkg.OPT_GEMV_SMALL_BATCH, 0)
    two = check_forward(prob, hidden, ids, wts, f"two launches M={M} ctas={num_ctas}")
    pkg.moe_w4a16_set_option(prob.moe.handle, pkg.OPT_GEMV_SMALL_BATCH, 1)
    assert_within_one_ulp(fused, two)
    prob.close()


def test_fused_small_batch_prepares_its_own_rows():
    # the fused launch routes, gathers and zeroes for itself and keeps its counters
    # in the handle: repeated calls (the counters cleared by each call's last CTA),
    # a bad expert id (the status bit, published in the workspace header), the
    # intermediate and accumulator read-back, and act-order weights (the gather in
    # the packing order) all behave as on the two-launch path
    E, K, N, k, M = 16, 512, 256, 4, 3
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    prob = Problem(E, K, N, k)
    h = prob.moe.handle
    pkg.moe_w4a16_set_option(h, pkg.OPT_FUSED_SMALL_BATCH, 1)
    try:
        for step in range(3):
            hidden, ids, wts = workload_inputs(wl, step=step)
            got = check_forward(prob, hidden, ids, wts, f"fused call {step}")
        inter = prob.moe.intermediate(M).cpu().numpy()
        acc = prob.moe.accumulator(M).cpu().numpy()
        pkg.moe_w4a16_set_option(h, pkg.OPT_FUSED_SMALL_BATCH, 0)
        pkg.moe_w4a16_set_option(h, pkg.OPT_GEMV_SMALL_BATCH, 0)  # (the tensor-core launches)
        two = check_forward(prob, hidden, ids, wts, "two launches")
        assert_within_one_ulp(got, two)
        # (the fused launch splits the gate/up steps at multiples of 4, so a split
        # unit's fp32 partial sums may add in another order: h to one fp16 unit)
        np.testing.assert_allclose(prob.moe.intermediate(M).cpu().numpy(), inter, rtol=2.0 ** -10,
                                   atol=2.0 ** -24 * float(np.abs(inter).max()))
        np.testing.assert_allclose(prob.moe.accumulator(M).cpu().numpy(), acc, rtol=1e-5,
                                   atol=1e-5 * float(np.abs(acc).max()))
        pkg.moe_w4a16_set_option(h, pkg.OPT_FUSED_SMALL_BATCH, 1)
        bad = ids.copy()
        bad[1, 2] = E + 5
        got = prob.run(hidden, bad, wts)
        assert prob.moe.status() == pkg.STATUS_BAD_EXPERT_ID
        assert_close(got, prob.reference(hidden, np.where(bad >= E, -1, bad), wts), "fused, bad id")
        check_forward(prob, hidden, ids, wts, "fused after a bad id")  # status clean again
    finally:
        prob.close()


def test_hot_expert_spans_several_token_tiles():
    # one expert receives every token (> 128 rows: several token tiles of one expert)
    E, K, N, k, M = 8, 768, 384, 2, 300
    prob = Problem(E, K, N, k)
    rng = np.random.default_rng(4)
    hidden = inputs.hidden_states(M, K)
    ids = np.stack([np.array([3, rng.choice([e for e in range(E) if e != 3])]) for _ in range(M)]).astype(np.int32)
    wts = rng.uniform(0.2, 0.8, size=(M, k)).astype(np.float32)
    for ctas in (None, 7):
        if ctas:
            prob.set_ctas(ctas)
        check_forward(prob, hidden, ids, wts, f"hot expert ctas={ctas}")
    prob.close()


@pytest.mark.parametrize("step_cost", [0, 1, 8, 64])
@pytest.mark.parametrize("num_ctas", [None, 5, 256])
def test_cost_weighted_stream_k_shares(step_cost, num_ctas):
    # Zipf-skewed routing gives token tiles of 1 to 4 row groups; the align kernel
    # then splits each GEMM's steps by cost, not by count (0 = even split). Every
    # split must give the oracle's result. (Two splits are not compared with each
    # other bit for bit: where a gate/up unit is cut moves the fp32 partial sums,
    # and a one-unit change in the bf16 intermediate carries into the output.)
    E, K, N, k, M = 16, 512, 256, 4, 300
    prob = Problem(E, K, N, k, num_ctas=num_ctas)
    rng = np.random.default_rng(11)
    ids = zipf_ids(rng, M, E, k, s=1.6)
    hidden = inputs.hidden_states(M, K)
    wts = rng.uniform(0.1, 1.0, size=(M, k)).astype(np.float32)
    wts /= wts.sum(axis=1, keepdims=True)
    pkg.moe_w4a16_set_option(prob.moe.handle, pkg.OPT_STEP_COST_GATEUP, step_cost)
    pkg.moe_w4a16_set_option(prob.moe.handle, pkg.OPT_STEP_COST_DOWN, (step_cost * 3) % 65)
    check_forward(prob, hidden, ids, wts, f"step cost {step_cost} ctas {num_ctas}")
    prob.close()


def test_bad_expert_ids_are_skipped_and_flagged():
    wl = inputs.WORKLOADS["tiny"]
    prob = Problem(wl.E, wl.K, wl.N, wl.topk)
    hidden, ids, wts = workload_inputs(wl)
    ids = ids.copy()
    ids[1, 0] = -3
    ids[2, 1] = wl.E
    got = prob.run(hidden, ids, wts)
    assert prob.moe.status() & pkg.STATUS_BAD_EXPERT_ID
    assert_close(got, prob.reference(hidden, ids, wts), "bad ids")
    prob.close()


def test_zero_tokens_and_small_workspace():
    wl = inputs.WORKLOADS["tiny"]
    prob = Problem(wl.E, wl.K, wl.N, wl.topk)
    h = prob.moe.handle
    empty = torch.zeros((0, wl.K), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    pkg.moe_w4a16_forward(h, empty, empty, empty, empty, 0, ws)  # M == 0 is a no-op
    hidden, ids, wts = workload_inputs(wl)
    out = torch.empty((wl.M, wl.K), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkg.MoeW4A16Error) as ei:
        pkg.moe_w4a16_forward(h, dev(bits16(hidden)), dev(ids), dev(wts), out, wl.M, ws)
    assert ei.value.code == -3
    prob.close()


def test_forward_host_matches_device_forward():
    E, K, N, k, M = 16, 512, 256, 4, 23
    prob = Problem(E, K, N, k)
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    hidden, ids, wts = workload_inputs(wl)
    dev_out = prob.run(hidden, ids, wts)
    h_hidden = torch.from_numpy(bits16(hidden)).pin_memory()
    h_ids = torch.from_numpy(ids).pin_memory()
    h_wts = torch.from_numpy(wts).pin_memory()
    h_out = torch.zeros((M, K), dtype=torch.int16).pin_memory()
    prob.moe.forward_host(h_hidden, h_ids, h_wts, h_out)
    host_out = h_out.view(torch.bfloat16).float().numpy().astype(np.float64)
    assert_close(host_out, prob.reference(hidden, ids, wts), "forward_host")
    assert_within_one_ulp(host_out, dev_out)
    prob.close()


def _host_forward(prob, hidden, ids, wts, pinned):
    M, K = hidden.shape
    bufs = [torch.from_numpy(bits16(hidden).copy()), torch.from_numpy(ids.copy()),
            torch.from_numpy(wts.copy()), torch.zeros((M, K), dtype=torch.int16)]
    if pinned:
        bufs = [t.pin_memory() for t in bufs]
    prob.moe.forward_host(*bufs)
    return bufs[3].view(torch.bfloat16).float().numpy().astype(np.float64)


def test_forward_host_zero_copy_and_staged_paths():
    # small batches read pinned caller buffers in place (zero-copy) or pass through
    # the handle's pinned staging when the buffers are pageable; large batches use
    # the copy engines: every route must give the device forward's result
    E, K, N, k = 16, 512, 256, 4
    prob = Problem(E, K, N, k)
    cases = [(1, True, 0), (1, False, 1), (3, True, 2), (3, False, 3), ("ctas", 7, 0), (2, True, 4),
             (2, False, 5), ("profile", 1, 0), (1, True, 6), (1, False, 7), ("profile", 0, 0),
             (1100, True, 8), (1100, False, 9), (1, False, 10)]
    for what, arg, seed in cases:
        if what == "ctas":
            prob.set_ctas(arg)
            continue
        if what == "profile":
            pkg.moe_w4a16_set_option(prob.moe.handle, pkg.OPT_PROFILE, arg)
            continue
        M = what
        wl = inputs.Workload("mid", E, K, N, k, M, "normal")
        hidden, ids, wts = workload_inputs(wl, step=seed)
        host_out = _host_forward(prob, hidden, ids, wts, pinned=arg)
        dev_out = prob.run(hidden, ids, wts)
        assert_within_one_ulp(host_out, dev_out)
        if M <= 3:
            assert_close(host_out, prob.reference(hidden, ids, wts), f"forward_host M={M} pinned={arg}")
    prob.close()


def test_forward_host_output_complete_on_return():
    # a host-buffer call returns with the output in the caller's buffer: filled
    # with NaNs before every call, it must hold the whole result as soon as the
    # call returns, call after call, pinned and pageable
    E, K, N, k = 16, 512, 256, 4
    prob = Problem(E, K, N, k)
    for step in range(12):
        M = 1 + step % 3
        pinned = step % 4 != 3
        wl = inputs.Workload("mid", E, K, N, k, M, "normal")
        hidden, ids, wts = workload_inputs(wl, step=step + 20)
        bufs = [torch.from_numpy(bits16(hidden).copy()), torch.from_numpy(ids.copy()), torch.from_numpy(wts.copy()),
                torch.full((M, K), 0x7FC0, dtype=torch.int16)]
        if pinned:
            bufs = [t.pin_memory() for t in bufs]
        prob.moe.forward_host(*bufs)
        host_bits = bufs[3].numpy().copy()  # read right after the return, before any other call
        assert prob.moe.status() == 0
        dev_out = prob.run(hidden, ids, wts)
        host_out = host_bits.view(np.uint16).astype(np.uint32) << 16
        host_out = host_out.view(np.float32).astype(np.float64)
        assert np.all(np.isfinite(host_out)), f"step {step}: output not complete on return"
        assert_within_one_ulp(host_out, dev_out)
    prob.close()


@pytest.mark.parametrize("M", [1, 37])
def test_forward_replays_from_a_cuda_graph(M):
    # the forward allocates nothing and makes no host-synchronising call, so it can
    # be captured once and replayed on new inputs copied into the same buffers
    E, K, N, k = 16, 512, 256, 4
    prob = Problem(E, K, N, k)
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    steps = [workload_inputs(wl, step=s) for s in range(3)]
    static = [dev(bits16(steps[0][0])), dev(steps[0][1]), dev(steps[0][2])]
    out = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    prob.moe.ensure_workspace(M)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        prob.moe.forward(*static, out=out)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        prob.moe.forward(*static, out=out)
    for s, (hidden, ids, wts) in enumerate(steps[1:] + steps[:1]):
        for dst, src in zip(static, (dev(bits16(hidden)), dev(ids), dev(wts))):
            dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        got = bf16_tensor_to_f64(out)
        assert prob.moe.status() == 0
        assert_within_one_ulp(got, prob.run(hidden, ids, wts))
        if s == 0:
            assert_close(got, prob.reference(hidden, ids, wts), f"graph replay M={M}")
    del g
    prob.close()


def test_repeated_calls_agree():
    E, K, N, k, M = 16, 512, 256, 4, 64
    prob = Problem(E, K, N, k)
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    hidden, ids, wts = workload_inputs(wl)
    a = prob.run(hidden, ids, wts)
    b = prob.run(hidden, ids, wts)
    # the down GEMM adds partial products with float atomics: only the summation
    # order may differ, which can flip the last bit of the bf16 output
    assert_within_one_ulp(a, b)
    prob.close()


# ---------------------------------------------------------------------------- router


@pytest.mark.parametrize("M,E,k,routing", [
    (1, 384, 8, "uniform"), (9, 384, 8, "normal"), (1024, 384, 8, "zipf"), (1024, 384, 8, "normal"),
    (37, 40, 5, "ties"), (5, 1024, 32, "normal"), (3, 7, 7, "normal"), (64, 33, 1, "ties"),
])
def test_router_matches_oracle(M, E, k, routing):
    # ids bit-exact (ties by ascending expert id), weights to fp32 rounding
    if routing == "ties":
        logits = (np.round(np.random.default_rng(M).standard_normal((M, E)) * 2) / 2).astype(np.float32)
    else:
        logits = inputs.router_logits(M, E, routing)
    ref_ids, ref_w = oracle.route(logits, k)
    d_ids = torch.full((M, k), -1, dtype=torch.int32, device="cuda")
    d_w = torch.full((M, k), -1.0, dtype=torch.float32, device="cuda")
    pkg.moe_w4a16_route(dev(logits), M, E, k, d_ids, d_w)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(d_ids.cpu().numpy(), ref_ids)
    np.testing.assert_allclose(d_w.cpu().numpy(), ref_w, rtol=2e-6, atol=1e-9)


@pytest.mark.parametrize("M", [1, 4, 37])
def test_forward_logits_routes_then_runs_the_forward(M):
    # M * k <= 32 routes inside the first launch, larger batches in a router launch
    E, K, N, k = 16, 512, 256, 8
    prob = Problem(E, K, N, k)
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    hidden, logits = inputs.workload_inputs(wl)
    ref_ids, ref_w = oracle.route(logits, k)
    out, d_ids, d_w = prob.moe.forward_logits(dev(bits16(hidden)), dev(logits))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(d_ids.cpu().numpy(), ref_ids)
    np.testing.assert_allclose(d_w.cpu().numpy(), ref_w, rtol=2e-6, atol=1e-9)
    got = bf16_tensor_to_f64(out)
    assert prob.moe.status() == 0
    assert_close(got, prob.reference(hidden, ref_ids, ref_w.astype(np.float32)), f"forward_logits M={M}")
    assert_within_one_ulp(got, prob.run(hidden, d_ids.cpu().numpy(), d_w.cpu().numpy()))
    prob.close()


# ---------------------------------------------------------------------------- fp16 operand range


@pytest.mark.parametrize("bad", [0x452B, 0xC52B, 0x4600, 0x3870, 0x0001, 0x7F80, 0x7FC0, 0xFF80])
def test_pack_rejects_unsupported_scales(bad):
    # 2736 and -2736 (just above the largest accepted magnitude: -24 * s leaves
    # fp16's range), 8192, just below 2^-14 (not exact in fp16), a subnormal, +inf,
    # NaN, -inf
    E, K, N = 2, 256, 128
    q1, s1, q2, s2 = inputs.all_expert_weights(E, K, N)
    s2 = s2.copy()
    s2[1, 3, 77] = bad
    moe = pkg.MoEW4A16(E, K, N, 2)
    with pytest.raises(pkg.MoeW4A16Error) as ei:
        moe.pack(dev(q1), dev(bits16(s1)), dev(q2), dev(bits16(s2)))
    assert ei.value.code == pkg.UNSUPPORTED_SCALE
    with pytest.raises(pkg.MoeW4A16Error) as ei:  # the handle stays unpacked
        moe.forward(dev(bits16(inputs.hidden_states(1, K))), dev(np.zeros((1, 2), np.int32)),
                    dev(np.full((1, 2), 0.5, np.float32)))
    assert ei.value.code == pkg.NOT_PACKED
    moe.close()


def test_boundary_scales_are_exact():
    # 0, -0 and 2^-14 (the smallest accepted magnitude) in the gate/up scales, 2720
    # and -2720 (the largest) in the down scales -- in the gate/up scales those
    # would only overflow the intermediate, whatever the format -- are accepted,
    # and the forward stays exact with them
    E, K, N, k, M = 4, 256, 128, 2, 6
    q1, s1, q2, s2 = inputs.all_expert_weights(E, K, N)
    s1, s2 = s1.copy(), s2.copy()
    rng = np.random.default_rng(9)
    for arr, vals in ((s1, [0x0000, 0x8000, 0x3880, 0xB880]), (s2, [0x452A, 0xC52A, 0x3880, 0x0000])):
        flat = arr.reshape(-1)
        idx = rng.choice(flat.size, size=40, replace=False)
        flat[idx] = np.array(vals * 10, dtype=np.uint16)
    prob = Problem(E, K, N, k, weights=(q1, s1, q2, s2))
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    hidden, ids, wts = workload_inputs(wl)
    got = prob.run(hidden, ids, wts)
    assert prob.moe.status() == 0
    assert_close(got, prob.reference(hidden, ids, wts), "boundary scales")
    prob.close()


def per_row_errors(got, ref):
    out = []
    for t in range(ref.shape[0]):
        r, g = ref[t], got[t]
        nr = np.linalg.norm(r)
        rms = np.sqrt(np.mean(r ** 2))
        out.append((np.linalg.norm(g - r) / nr, np.max(np.abs(g - r)) / rms) if nr > 0 else (0.0, 0.0))
    return out


@pytest.mark.parametrize("M", [3, 12])
def test_hidden_rows_far_outside_fp16_range(M):
    # every token row is fed in at a power-of-two prescale chosen from its own largest
    # magnitude: rows from 1e-15 to 1e15 (fp16 covers 6e-5 .. 65504) all match the
    # oracle row by row; M = 3 (12 slots) takes the small-batch gather, M = 12 the
    # general one
    E, K, N, k = 8, 512, 256, 4
    prob = Problem(E, K, N, k)
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    hidden, ids, wts = workload_inputs(wl)
    x = oracle.bf16_to_f64(hidden).astype(np.float32)
    factors = np.array([1e6, 1e-6, 3e4, 1e15, 1e-15, 0.0, 1.0, 7e10, 2e-9, 65504.0, 1e5, 1e-4])[:M]
    x = (x * factors[:, None].astype(np.float32)).astype(np.float32)
    big = inputs.f32_to_bf16_bits(x)
    got = prob.run(big, ids, wts)
    ref = prob.reference(big, ids, wts)
    assert prob.moe.status() == 0
    assert np.all(np.isfinite(got))
    for t, (rel, mx) in enumerate(per_row_errors(got, ref)):
        if factors[t] == 0.0:
            assert np.all(got[t] == 0.0)
            continue
        assert rel <= 5e-3 and mx <= 2e-2, f"row {t} (scale {factors[t]:g}): rel {rel:.3e} max/rms {mx:.3e}"
    prob.close()


def test_intermediate_saturation_sets_status():
    # gate/up scales of 2720 make SiLU(g) * u far exceed fp16's range even for
    # prescaled rows: the epilogue saturates and says so; a normal call is clean again
    E, K, N, k, M = 4, 256, 128, 2, 3
    q1, s1, q2, s2 = inputs.all_expert_weights(E, K, N)
    hot = np.full_like(s1, 0x452A)
    prob = Problem(E, K, N, k, weights=(q1, hot, q2, s2))
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    hidden, ids, wts = workload_inputs(wl)
    prob.run(hidden, ids, wts)
    assert prob.moe.status() & pkg.STATUS_H_SATURATED
    prob.close()
    prob = Problem(E, K, N, k, weights=(q1, s1, q2, s2))
    check_forward(prob, hidden, ids, wts, "after saturation")
    prob.close()


# ---------------------------------------------------------------------------- give-up path


@pytest.mark.parametrize("M", [4, 40])
def test_wait_limit_gives_up_cleanly(M):
    # Each GEMM's epilogue is made to wait on a barrier that nothing ever arrives on,
    # with a 1 ms limit: the wait gives up, the kernels flag MOE_W4A16_STATUS_TIMEOUT,
    # every role stops at its next wait, in-flight copies and MMAs land, tensor
    # memory is freed and the call returns. The next call on the same handle, with
    # the hook off and the default limit, is clean and correct.
    E, K, N, k = 8, 512, 256, 4
    prob = Problem(E, K, N, k)
    wl = inputs.Workload("mid", E, K, N, k, M, "normal")
    hidden, ids, wts = workload_inputs(wl)
    h = prob.moe.handle
    pkg.moe_w4a16_set_option(h, pkg.OPT_WAIT_LIMIT_US, 1000)
    pkg.moe_w4a16_set_option(h, pkg.OPT_TEST_WAIT_NEVER_COMPLETES, 1)
    prob.run(hidden, ids, wts)  # returns; its output is not meaningful
    assert prob.moe.status() & pkg.STATUS_TIMEOUT
    if M * k <= 32:  # and the same through the fused small-batch launch
        pkg.moe_w4a16_set_option(h, pkg.OPT_FUSED_SMALL_BATCH, 1)
        prob.run(hidden, ids, wts)
        assert prob.moe.status() & pkg.STATUS_TIMEOUT
        pkg.moe_w4a16_set_option(h, pkg.OPT_FUSED_SMALL_BATCH, 0)
    pkg.moe_w4a16_set_option(h, pkg.OPT_TEST_WAIT_NEVER_COMPLETES, 0)
    pkg.moe_w4a16_set_option(h, pkg.OPT_WAIT_LIMIT_US, 0)
    check_forward(prob, hidden, ids, wts, f"after give-up M={M}")
    prob.close()


# ---------------------------------------------------------------------------- duplicate experts


@pytest.mark.parametrize("M", [3, 40])
def test_forward_with_duplicate_experts_in_a_token(M):
    # a token may name one expert in several of its slots: each slot is an
    # independent routed row (its own weight), as the oracle defines
    E, K, N, k = 6, 512, 256, 4
    prob = Problem(E, K, N, k)
    rng = np.random.default_rng(M)
    ids = rng.integers(0, E, size=(M, k)).astype(np.int32)
    ids[0] = [2, 2, 2, 5]
    ids[1] = [1, 1, 4, 4]
    hidden = inputs.hidden_states(M, K)
    wts = rng.uniform(0.1, 1.0, size=(M, k)).astype(np.float32)
    check_forward(prob, hidden, ids, wts, f"duplicates M={M}")
    prob.close()
