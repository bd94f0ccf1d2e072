"""The allocation-free forward (moe_w4a16_forward_noalloc) against the regular
one.

Some callers cannot allocate device memory for a workspace: a runtime that owns
every byte of the GPU through its own pool, a process whose device memory budget
is already committed, or a plug-in that must not call the host application's
allocator. The allocation-free entry point serves them with a fixed array inside
the library. These checks call it through the C-ABI twice in a row on different
inputs (the array keeps the previous call's contents, which must not matter) and
compare with moe_w4a16_forward on the same inputs, within the tolerances of the
other GPU tests. The file is named so that pytest collects it last."""
import numpy as np
import pytest
import torch

import int4_weight_only_moe_gb300 as pkg
from int4_weight_only_moe_gb300 import inputs
from tests.gpu_helpers import Problem, assert_close, bf16_tensor_to_f64, bits16, dev, workload_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def run_both(prob, wl, step):
    hidden, ids, wts = workload_inputs(wl, step=step)
    d_h, d_ids, d_w = dev(bits16(hidden)), dev(ids), dev(wts)
    ref = prob.moe.forward(d_h, d_ids, d_w)
    out = torch.full((wl.M, wl.K), float("nan"), dtype=torch.bfloat16, device="cuda")
    pkg.moe_w4a16_forward_noalloc(prob.moe.handle, d_h, d_ids, d_w, out, wl.M)
    torch.cuda.synchronize()
    got, want = bf16_tensor_to_f64(out), bf16_tensor_to_f64(ref)
    return got, want, prob.reference(hidden, ids, wts)


def within_one_ulp(a, b):
    # One bf16 unit of the larger value, plus the term by which two orders of the
    # down projection's float atomic additions can differ near zero (2^-16 of the
    # output's largest magnitude), as in the other GPU tests.
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(a), np.abs(b)) + 1e-30)) - 7)
    floor = np.exp2(-16.0) * max(float(np.abs(b).max()), 1e-30)
    return bool(np.all(np.abs(a - b) <= ulp + floor))


@pytest.mark.parametrize("shape", [(16, 512, 256, 4, 37), (48, 7168, 2048, 8, 1), (48, 7168, 2048, 8, 9)])
def test_noalloc_matches_forward_on_consecutive_calls(shape):
    E, K, N, k, M = shape
    prob = Problem(E, K, N, k)
    wl = inputs.Workload("noalloc", E, K, N, k, M, "normal")
    for step in (0, 1):  # two calls in a row, different inputs
        got, want, oracle_ref = run_both(prob, wl, step)
        assert np.all(np.isfinite(got))
        assert_close(got, want, f"noalloc vs forward {shape} call {step}")
        assert within_one_ulp(got, want), f"noalloc vs forward {shape} call {step}"
        assert_close(got, oracle_ref, f"noalloc vs oracle {shape} call {step}")
    prob.close()


def test_noalloc_rejects_batches_beyond_its_array():
    E, K, N, k = 48, 7168, 2048, 8
    moe = pkg.MoEW4A16(E, K, N, k)
    M = 1
    while pkg.moe_w4a16_workspace_size(moe.handle, M) <= pkg.NOALLOC_WORKSPACE_BYTES:
        M += 1
    hidden = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((M, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((M, k), dtype=torch.float32, device="cuda")
    out = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkg.MoeW4A16Error) as ei:
        pkg.moe_w4a16_forward_noalloc(moe.handle, hidden, ids, w, out, M)
    assert ei.value.code == pkg.WORKSPACE_TOO_SMALL
    assert "static array" in str(ei.value)
    moe.close()
