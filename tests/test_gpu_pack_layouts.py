"""The two other weight inputs of the repack: the compressed-tensors layout
(every output feature's reduction row contiguous) and GPTQ quantised in
activation order (a group index per reduction element), alone and together.
Each is checked bit for bit through the inverse repack, and end to end against
the oracle's own decoders of those layouts (oracle.dequantize_ct,
oracle.dequantize_g_idx) on the batched path and on the small-batch path, at a
mid size (several row tiles, k-blocks and token tiles) and at full size for a
decode step."""
import numpy as np
import pytest
import torch

import int4_weight_only_moe_gb300 as pkg
import oracle
from int4_weight_only_moe_gb300 import inputs
from tests.conftest import MARGINS
from tests.gpu_helpers import (assert_close, bf16_tensor_to_f64, bits16, check_accumulator, dev,
                               errors, workload_inputs)

pytestmark = pytest.mark.gpu

MID = inputs.Workload("layouts", 16, 512, 256, 4, 37, "normal")


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


class LayoutProblem:
    """Seeded weights of E experts in one layout, optionally in act order."""

    def __init__(self, E, K, N, topk, ct, act1, act2):
        self.E, self.K, self.N, self.ct = E, K, N, ct
        gen = inputs.expert_weights_ct if ct else inputs.expert_weights
        self.w = None
        for e in range(E):  # filled in place: no second host copy at full size
            ws = gen(e, K, N)
            if self.w is None:
                self.w = [np.empty((E,) + a.shape, a.dtype) for a in ws]
            for dst, a in zip(self.w, ws):
                dst[e] = a
        self.g1 = np.stack([inputs.act_order_g_idx(e, K, 0) for e in range(E)]) if act1 else None
        self.g2 = np.stack([inputs.act_order_g_idx(e, N, 1) for e in range(E)]) if act2 else None
        self.moe = pkg.MoEW4A16(E, K, N, topk)
        q1, s1, q2, s2 = self.w
        self.moe.pack(dev(q1), dev(bits16(s1)), dev(q2), dev(bits16(s2)),
                      layout=pkg.LAYOUT_COMPRESSED_TENSORS if ct else pkg.LAYOUT_GPTQ,
                      w1_g_idx=None if self.g1 is None else dev(self.g1),
                      w2_g_idx=None if self.g2 is None else dev(self.g2))
        torch.cuda.synchronize()

    def dense(self, e):
        q1, s1, q2, s2 = (a[e] for a in self.w)
        if self.ct:
            return oracle.dequantize_ct(q1, s1), oracle.dequantize_ct(q2, s2)
        d1 = (oracle.dequantize(q1, s1) if self.g1 is None else oracle.dequantize_g_idx(q1, s1, self.g1[e]))
        d2 = (oracle.dequantize(q2, s2) if self.g2 is None else oracle.dequantize_g_idx(q2, s2, self.g2[e]))
        return d1, d2

    def reference(self, hidden, ids, wts, tokens=None):
        return oracle.moe_forward(hidden, ids, wts, None, None, None, None, tokens=tokens,
                                  dense_source=self.dense)

    def close(self):
        self.moe.close()


CASES = [
    ("compressed-tensors", True, False, False),
    ("act-order w1+w2", False, True, True),
    ("act-order w1", False, True, False),
    ("act-order w2", False, False, True),
]


@pytest.mark.parametrize("name,ct,act1,act2", CASES)
def test_inverse_repack_is_bit_exact(name, ct, act1, act2):
    need_gpu()
    wl = MID
    p = LayoutProblem(wl.E, wl.K, wl.N, wl.topk, ct, act1, act2)
    try:
        outs = [torch.empty_like(dev(a)) for a in (p.w[0], bits16(p.w[1]), p.w[2], bits16(p.w[3]))]
        pkg.moe_w4a16_unpack_debug(p.moe.handle, *outs)
        torch.cuda.synchronize()
        for want, got, nm in zip(p.w, outs, ("w1_q", "w1_s", "w2_q", "w2_s")):
            np.testing.assert_array_equal(got.cpu().numpy().view(want.dtype), want, err_msg=f"{name} {nm}")
    finally:
        p.close()


@pytest.mark.parametrize("name,ct,act1,act2", CASES)
@pytest.mark.parametrize("M,fused", [(37, 0), (3, 0), (3, 1)])
def test_forward_matches_oracle_decoder(name, ct, act1, act2, M, fused):
    # M = 37: the batched path (align, gather, split token tiles); M = 3: the
    # small-batch path (routing and gather in one launch), or the fused launch
    # that gathers (in w1's packing order) for itself
    need_gpu()
    wl = MID
    p = LayoutProblem(wl.E, wl.K, wl.N, wl.topk, ct, act1, act2)
    pkg.moe_w4a16_set_option(p.moe.handle, pkg.OPT_FUSED_SMALL_BATCH, fused)
    try:
        hidden, ids, wts = workload_inputs(wl, M=M, step=M)
        out = p.moe.forward(dev(bits16(hidden)), dev(ids), dev(wts))
        torch.cuda.synchronize()
        got = bf16_tensor_to_f64(out)
        assert p.moe.status() == 0
        ref = p.reference(hidden, ids, wts)
        rel, mx = assert_close(got, ref, f"{name}, M={M}")
        acc = p.moe.accumulator(M).cpu().numpy().astype(np.float64)
        check_accumulator(acc, out.view(torch.int16).cpu().numpy(), ref, f"{name}, M={M}")
        MARGINS.append(f"pack layout {name}, M={M}{' fused' if fused else ''}: rel L2 {rel:.3e}, "
                       f"max|d|/rms {mx:.3e}")
    finally:
        p.close()


def test_act_order_intermediate_is_in_w2_packing_order():
    need_gpu()
    wl = MID
    p = LayoutProblem(wl.E, wl.K, wl.N, wl.topk, False, True, True)
    try:
        M = 5
        hidden, ids, wts = workload_inputs(wl, M=M, step=11)
        p.moe.forward(dev(bits16(hidden)), dev(ids), dev(wts))
        torch.cuda.synchronize()
        h_rows = p.moe.intermediate(M).cpu().numpy().astype(np.float64)
        x = oracle.bf16_to_f64(hidden)
        for t in range(M):
            for j in range(wl.topk):
                e = int(ids[t, j])
                w1, _ = p.dense(e)
                ref = oracle.expert_hidden(x[t:t + 1], w1)[0]
                order = np.argsort(p.g2[e], kind="stable")  # w2's packing order
                assert_close(h_rows[t * wl.topk + j][None, :], ref[order][None, :],
                             f"intermediate token {t} slot {j}", bf16_output=False)
    finally:
        p.close()


def test_bad_group_indices_are_rejected():
    need_gpu()
    E, K, N, k = 2, 256, 128, 2
    ws = [inputs.expert_weights(e, K, N) for e in range(E)]
    q1, s1, q2, s2 = (np.stack([w[i] for w in ws]) for i in range(4))
    q1, s1, q2, s2 = dev(q1), dev(bits16(s1)), dev(q2), dev(bits16(s2))
    good1 = np.stack([inputs.act_order_g_idx(e, K, 0) for e in range(E)])
    moe = pkg.MoEW4A16(E, K, N, k)
    try:
        bad_cases = []
        b = good1.copy()
        b[1, 5] = K // 32  # out of range
        bad_cases.append(b)
        b = good1.copy()
        b[0, np.nonzero(b[0] == 0)[0][0]] = 1  # group 0 has 31 members, group 1 has 33
        bad_cases.append(b)
        b = good1.copy()
        b[0, 0] = -1
        bad_cases.append(b)
        for b in bad_cases:
            with pytest.raises(pkg.MoeW4A16Error) as ei:
                moe.pack(q1, s1, q2, s2, w1_g_idx=dev(b))
            assert ei.value.code == pkg.BAD_G_IDX
            # the handle stays unpacked
            hidden, ids, wts = workload_inputs(inputs.Workload("x", E, K, N, k, 2, "normal"))
            with pytest.raises(pkg.MoeW4A16Error) as ei:
                moe.forward(dev(bits16(hidden)), dev(ids), dev(wts))
            assert ei.value.code == pkg.NOT_PACKED
        moe.pack(q1, s1, q2, s2, w1_g_idx=dev(good1))  # and a good one still packs
    finally:
        moe.close()


def test_full_size_decode_compressed_tensors_and_act_order():
    # decode at the benchmark's dimensions with act-order weights: the gather's
    # permuted copy of a 7168-element row and both permuted GEMMs
    need_gpu()
    wl = inputs.WORKLOADS["decode"]
    hidden, ids, wts = workload_inputs(wl, step=5)
    for ct, act in ((True, False), (False, True)):
        p = LayoutProblem(wl.E, wl.K, wl.N, wl.topk, ct, act, act)
        try:
            out = p.moe.forward(dev(bits16(hidden)), dev(ids), dev(wts))
            torch.cuda.synchronize()
            assert p.moe.status() == 0
            got = bf16_tensor_to_f64(out)
            ref = p.reference(hidden, ids, wts)
            rel, mx = assert_close(got, ref, f"full-size decode ct={ct} act={act}")
            MARGINS.append(f"full-size decode, {'compressed-tensors' if ct else 'act-order'}: "
                           f"rel L2 {rel:.3e}, max|d|/rms {mx:.3e}")
        finally:
            p.close()
