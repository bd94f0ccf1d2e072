"""Shared helpers of the GPU parity tests: upload seeded inputs, run the CUDA path
through the C-ABI binding, and compare with the CPU oracle."""
import numpy as np
import torch

import int4_weight_only_moe_gb300 as pkg
import oracle
from int4_weight_only_moe_gb300 import inputs

# Floating-point tolerance of the fused forward against the float64 oracle
# (relative L2 error, and largest absolute error relative to the reference RMS).
TOL_REL_L2 = 5e-3
TOL_MAX_OVER_RMS = 2e-2
# The output is bf16: rounding the exact result to bf16 alone moves an element by
# up to half a unit in the last place, 2^-8 of its magnitude, which for an element
# beyond about 5 times the RMS exceeds TOL_MAX_OVER_RMS whatever the computation.
# The bf16 output's largest error is therefore bounded by the tolerance plus that
# rounding term; the unrounded fp32 accumulator is held to the tolerance itself
# (check_accumulator), and the output must be its exact rounding.
BF16_HALF_ULP_REL = 2.0 ** -8


def errors(got, ref):
    d = got - ref
    nref = np.linalg.norm(ref)
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    rel = np.linalg.norm(d) / nref if nref > 0 else np.linalg.norm(d)
    mx = np.max(np.abs(d)) / rms if rms > 0 else np.max(np.abs(d), initial=0.0)
    return float(rel), float(mx)


def excess_over_rounding(got, ref):
    """Largest error beyond the bf16 rounding of the reference, over the reference RMS."""
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    ex = np.max(np.abs(got - ref) - BF16_HALF_ULP_REL * np.abs(ref), initial=0.0)
    return float(ex / rms) if rms > 0 else float(ex)


def assert_close(got, ref, what="", bf16_output=True):
    """``got`` within the tolerance of ``ref``; for a bf16 output the largest-error
    bound also admits the output's own rounding (see BF16_HALF_ULP_REL)."""
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rel, mx = errors(got, ref)
    ex = excess_over_rounding(got, ref) if bf16_output else mx
    assert rel <= TOL_REL_L2 and ex <= TOL_MAX_OVER_RMS, (
        f"{what}: rel L2 {rel:.3e} (limit {TOL_REL_L2}), max|d|/rms {mx:.3e}, beyond bf16 rounding "
        f"{ex:.3e} (limit {TOL_MAX_OVER_RMS})")
    return rel, mx


def check_accumulator(acc, out, ref, what=""):
    """The fp32 accumulator (before rounding) meets the tolerance itself, and the bf16
    output is its round-to-nearest-even, bit for bit."""
    from int4_weight_only_moe_gb300 import inputs
    rel, mx = errors(acc, ref)
    assert rel <= TOL_REL_L2 and mx <= TOL_MAX_OVER_RMS, (
        f"{what} fp32 accumulator: rel L2 {rel:.3e}, max|d|/rms {mx:.3e}")
    want = inputs.f32_to_bf16_bits(acc.astype(np.float32))
    np.testing.assert_array_equal(np.ascontiguousarray(out).view(np.uint16), want)
    return rel, mx


def workload_inputs(wl, step=0, M=None):
    """Seeded hidden states of ``wl`` and their routing by the oracle's router:
    (hidden bf16 bits, topk_ids int32, topk_weights float32)."""
    hidden, logits = inputs.workload_inputs(wl, step=step, M=M)
    ids, w = oracle.route(logits, wl.topk)
    return hidden, ids, w.astype(np.float32)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits16(a):
    return np.ascontiguousarray(a).view(np.int16)


def bf16_tensor_to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


class Problem:
    """A handle with packed seeded weights, plus the host copy the oracle reads."""

    def __init__(self, E, K, N, topk, weights=None, num_ctas=None):
        self.E, self.K, self.N, self.topk = E, K, N, topk
        self.w = weights if weights is not None else inputs.all_expert_weights(E, K, N)
        self.moe = pkg.MoEW4A16(E, K, N, topk)
        if num_ctas is not None:
            pkg.moe_w4a16_set_option(self.moe.handle, pkg.OPT_NUM_CTAS, num_ctas)
        q1, s1, q2, s2 = self.w
        d = [dev(q1), dev(bits16(s1)), dev(q2), dev(bits16(s2))]
        self.moe.pack(*d)
        torch.cuda.synchronize()
        del d

    def set_ctas(self, n):
        pkg.moe_w4a16_set_option(self.moe.handle, pkg.OPT_NUM_CTAS, n)

    def run(self, hidden, ids, wts):
        out = self.moe.forward(dev(bits16(hidden)), dev(ids), dev(wts))
        torch.cuda.synchronize()
        return bf16_tensor_to_f64(out)

    def reference(self, hidden, ids, wts, tokens=None):
        return oracle.moe_forward(hidden, ids, wts, *self.w, tokens=tokens)

    def close(self):
        self.moe.close()
