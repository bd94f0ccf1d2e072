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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits16(a):
    return np.ascontiguousarray(a).view(np.int16)


def errors(got, ref):
    d = got - ref
    nref = np.linalg.norm(ref)
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    rel = np.linalg.norm(d) / nref if nref > 0 else np.linalg.norm(d)
    mx = np.max(np.abs(d)) / rms if rms > 0 else np.max(np.abs(d), initial=0.0)
    return float(rel), float(mx)


def assert_close(got, ref, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rel, mx = errors(got, ref)
    assert rel <= TOL_REL_L2 and mx <= TOL_MAX_OVER_RMS, (
        f"{what}: rel L2 {rel:.3e} (limit {TOL_REL_L2}), max|d|/rms {mx:.3e} (limit {TOL_MAX_OVER_RMS})")
    return rel, mx


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
