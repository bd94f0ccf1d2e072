"""Expert-parallel handles on one GPU: the layer's experts split into G
contiguous ranges, one handle per range, each forward_partial over its own
experts; the partials' sum (on one GPU a plain device add stands in for the
ranks' all-reduce) rounded by finalize must match the oracle's full layer, and
the sum must round to the output bit for bit. Slots of other ranges are skipped
without a status bit; ids outside the layer still raise it."""
import numpy as np
import pytest
import torch

import int4_weight_only_moe_gb300 as pkg
import oracle
from int4_weight_only_moe_gb300 import ep, inputs
from tests.conftest import MARGINS
from tests.gpu_helpers import (assert_close, bf16_tensor_to_f64, bits16, check_accumulator, dev,
                               workload_inputs)

pytestmark = pytest.mark.gpu

MID = inputs.Workload("ep", 16, 512, 256, 4, 37, "normal")


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def expert_slice(E, K, N, b, e):
    ws = [inputs.expert_weights(x, K, N) for x in range(b, e)]
    return [np.stack([w[i] for w in ws]) for i in range(4)]


def rank_handles(wl, world):
    hs = []
    for r in range(world):
        b, e = ep.expert_range(wl.E, world, r)
        moe = pkg.MoEW4A16(wl.E, wl.K, wl.N, wl.topk, expert_range=(b, e))
        q1, s1, q2, s2 = expert_slice(wl.E, wl.K, wl.N, b, e)
        moe.pack(dev(q1), dev(bits16(s1)), dev(q2), dev(bits16(s2)))
        hs.append(moe)
    torch.cuda.synchronize()
    return hs


def ep_run(hs, hidden, ids, wts):
    x, i, w = dev(bits16(hidden)), dev(ids), dev(wts)
    total = None
    for moe in hs:
        part = moe.forward_partial(x, i, w)
        total = part.clone() if total is None else total + part
    out = ep.finalize(total)
    torch.cuda.synchronize()
    return total, out


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("M,fused", [(37, 0), (3, 0), (3, 1)])
def test_partials_sum_to_the_layer(world, M, fused):
    need_gpu()
    wl = MID
    hs = rank_handles(wl, world)
    for moe in hs:
        pkg.moe_w4a16_set_option(moe.handle, pkg.OPT_FUSED_SMALL_BATCH, fused)
    try:
        hidden, ids, wts = workload_inputs(wl, M=M, step=world)
        total, out = ep_run(hs, hidden, ids, wts)
        for moe in hs:
            assert moe.status() == 0  # other ranges' slots are skipped silently
        ref = oracle.moe_forward(hidden, ids, wts, *inputs.all_expert_weights(wl.E, wl.K, wl.N))
        got = bf16_tensor_to_f64(out)
        rel, mx = assert_close(got, ref, f"EP world {world}, M={M}")
        check_accumulator(total.cpu().numpy().astype(np.float64), out.view(torch.int16).cpu().numpy(), ref,
                          f"EP world {world}, M={M}")
        MARGINS.append(f"expert-parallel world {world}, M={M}{' fused' if fused else ''}: rel L2 {rel:.3e}, "
                       f"max|d|/rms {mx:.3e}")
    finally:
        for moe in hs:
            moe.close()


def test_ids_outside_the_layer_are_flagged():
    need_gpu()
    wl = MID
    hs = rank_handles(wl, 2)
    try:
        for M in (37, 3):
            hidden, ids, wts = workload_inputs(wl, M=M, step=7)
            ids = ids.copy()
            ids[0, 0] = wl.E  # no expert of the layer
            total, _ = ep_run(hs, hidden, ids, wts)
            assert all(moe.status() == pkg.STATUS_BAD_EXPERT_ID for moe in hs)
            ref_ids = np.where(ids == wl.E, -1, ids)
            ref = oracle.moe_forward(hidden, ref_ids, wts, *inputs.all_expert_weights(wl.E, wl.K, wl.N))
            assert_close(total.cpu().numpy().astype(np.float64), ref, "EP with a bad id", bf16_output=False)
    finally:
        for moe in hs:
            moe.close()


def test_router_of_a_part_sees_every_expert():
    need_gpu()
    wl = MID
    hs = rank_handles(wl, 2)
    try:
        _, logits = inputs.workload_inputs(wl, M=9)
        want, _ = oracle.route(logits, wl.topk)
        for moe in hs:
            ids, _ = moe.route(dev(logits))
            np.testing.assert_array_equal(ids.cpu().numpy(), want)
    finally:
        for moe in hs:
            moe.close()


def test_full_size_decode_two_parts():
    need_gpu()
    wl = inputs.WORKLOADS["decode"]
    hidden, ids, wts = workload_inputs(wl, step=9)
    hs = rank_handles(wl, 2)
    try:
        total, out = ep_run(hs, hidden, ids, wts)
        assert all(moe.status() == 0 for moe in hs)

        def source(e):
            return inputs.expert_weights(e, wl.K, wl.N)

        ref = oracle.moe_forward(hidden, ids, wts, None, None, None, None, expert_source=source)
        rel, mx = assert_close(bf16_tensor_to_f64(out), ref, "full-size decode, 2 parts")
        MARGINS.append(f"expert-parallel full-size decode, 2 parts: rel L2 {rel:.3e}, max|d|/rms {mx:.3e}")
    finally:
        for moe in hs:
            moe.close()
