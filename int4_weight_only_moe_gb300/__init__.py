"""INT4 weight-only (W4A16) fused Mixture-of-Experts feed-forward for GB300.

Thin Python binding of the C-ABI library ``libmoe_w4a16.so`` (declared in
``include/moe_w4a16.h``). The functions below carry the same names as the C
entry points and only marshal arguments: torch tensors provide device memory
and streams, every step of the computation runs in the library's CUDA kernels.
There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "MoeW4A16Error", "lib", "moe_w4a16_create", "moe_w4a16_destroy", "moe_w4a16_pack",
    "moe_w4a16_pack_ex", "LAYOUT_GPTQ", "LAYOUT_COMPRESSED_TENSORS", "BAD_G_IDX",
    "moe_w4a16_create_ep", "moe_w4a16_forward_partial", "moe_w4a16_finalize",
    "moe_w4a16_workspace_size", "moe_w4a16_host_staging_size", "moe_w4a16_forward",
    "moe_w4a16_forward_host", "moe_w4a16_status", "moe_w4a16_last_error",
    "moe_w4a16_set_option", "moe_w4a16_kernel_times", "moe_w4a16_packed_bytes",
    "moe_w4a16_align_debug", "moe_w4a16_unpack_debug", "moe_w4a16_read_intermediate",
    "moe_w4a16_schedule_debug", "moe_w4a16_read_accumulator", "moe_w4a16_route", "moe_w4a16_forward_logits", "moe_w4a16_forward_noalloc", "NOALLOC_WORKSPACE_BYTES", "MoEW4A16",
    "OPT_NUM_CTAS", "OPT_PROFILE", "OPT_PDL", "OPT_STEP_COST_GATEUP", "OPT_STEP_COST_DOWN",
    "OPT_WAIT_LIMIT_US", "OPT_TEST_WAIT_NEVER_COMPLETES", "OPT_FUSED_SMALL_BATCH", "OPT_GEMV_SMALL_BATCH", "OPT_GEMV_ONE_LAUNCH", "STATUS_BAD_EXPERT_ID", "STATUS_TIMEOUT", "STATUS_H_SATURATED",
    "STATUS_BAD_SCHEDULE",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libmoe_w4a16.so")

OK, INVALID_ARG, UNSUPPORTED_SHAPE, WORKSPACE_TOO_SMALL, CUDA_ERROR, NOT_PACKED = 0, -1, -2, -3, -4, -5
UNSUPPORTED_SCALE, BAD_G_IDX = -6, -7
LAYOUT_GPTQ, LAYOUT_COMPRESSED_TENSORS = 0, 1
STATUS_BAD_EXPERT_ID, STATUS_TIMEOUT, STATUS_H_SATURATED, STATUS_BAD_SCHEDULE = 1, 2, 4, 16
OPT_NUM_CTAS, OPT_PROFILE, OPT_PDL = 1, 2, 3
OPT_STEP_COST_GATEUP, OPT_STEP_COST_DOWN, OPT_WAIT_LIMIT_US = 4, 5, 6
OPT_TEST_WAIT_NEVER_COMPLETES = 7
OPT_FUSED_SMALL_BATCH = 8
OPT_GEMV_SMALL_BATCH = 9
OPT_GEMV_ONE_LAUNCH = 10
NOALLOC_WORKSPACE_BYTES = 48 << 20

_c_int, _c_size, _vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p

# name -> (restype, argtypes); mirrors include/moe_w4a16.h
_SIGNATURES = {
    "moe_w4a16_create": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, ctypes.POINTER(_vp)]),
    "moe_w4a16_destroy": (_c_int, [_vp]),
    "moe_w4a16_pack": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp]),
    "moe_w4a16_pack_ex": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _vp, _vp, _vp]),
    "moe_w4a16_create_ep": (_c_int, [_c_int] * 7 + [ctypes.POINTER(_vp)]),
    "moe_w4a16_forward_partial": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_size, _vp]),
    "moe_w4a16_finalize": (_c_int, [_vp, _vp, ctypes.c_longlong, _vp]),
    "moe_w4a16_workspace_size": (_c_size, [_vp, _c_int]),
    "moe_w4a16_host_staging_size": (_c_size, [_vp, _c_int]),
    "moe_w4a16_forward": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_size, _vp]),
    "moe_w4a16_forward_host": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_size, _vp]),
    "moe_w4a16_route": (_c_int, [_vp, _c_int, _c_int, _c_int, _vp, _vp, _vp]),
    "moe_w4a16_forward_logits": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_size, _vp]),
    "moe_w4a16_status": (_c_int, [_vp, _vp, ctypes.POINTER(ctypes.c_int32), _vp]),
    "moe_w4a16_last_error": (ctypes.c_char_p, []),
    "moe_w4a16_set_option": (_c_int, [_vp, _c_int, _c_int]),
    "moe_w4a16_kernel_times": (_c_int, [_vp, ctypes.POINTER(ctypes.c_float), _c_int]),
    "moe_w4a16_packed_bytes": (_c_size, [_vp]),
    "moe_w4a16_align_debug": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp, _c_int, _vp]),
    "moe_w4a16_unpack_debug": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp]),
    "moe_w4a16_read_intermediate": (_c_int, [_vp, _vp, _c_int, _vp, _vp]),
    "moe_w4a16_read_accumulator": (_c_int, [_vp, _vp, _c_int, _vp, _vp]),
    "moe_w4a16_schedule_debug": (_c_int, [_vp, _vp, _c_int, ctypes.POINTER(ctypes.c_int64), _c_int,
                                          ctypes.POINTER(_c_int), _vp]),
    "moe_w4a16_forward_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _vp]),
}

_LIB = None


class MoeW4A16Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"moe_w4a16 error {code}: {msg}")
        self.code = code


def lib() -> ctypes.CDLL:
    """Load the library (it must have been built; see ``__graft_entry__.build``)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def moe_w4a16_last_error() -> str:
    return lib().moe_w4a16_last_error().decode()


def _check(rc: int):
    if rc != OK:
        raise MoeW4A16Error(rc, moe_w4a16_last_error())
    return rc


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:  # the current stream's handle without building a Stream object
            return int(raw(torch.cuda.current_device()))
        return int(torch.cuda.current_stream().cuda_stream)
    return int(getattr(stream, "cuda_stream", stream))


_DTYPES: dict = {}


def _dtypes(names):
    d = _DTYPES.get(names)
    if d is None:
        import torch
        d = _DTYPES[names] = tuple(getattr(torch, n) for n in names if hasattr(torch, n))
    return d


def _need(t, dtype_names, shape, name, device=True):
    if t.shape != shape:
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype not in _dtypes(dtype_names):
        raise ValueError(f"{name}: dtype {t.dtype}, expected one of {dtype_names}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not device and t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")


_BITS16 = ("bfloat16", "int16", "uint16")


def moe_w4a16_create(E: int, K: int, N: int, topk: int, group_size: int = 32) -> int:
    h = _vp()
    _check(lib().moe_w4a16_create(E, K, N, topk, group_size, ctypes.byref(h)))
    return h.value


def moe_w4a16_create_ep(E_total, expert_begin, expert_end, K, N, topk, group_size=32) -> int:
    h = _vp()
    _check(lib().moe_w4a16_create_ep(E_total, expert_begin, expert_end, K, N, topk, group_size,
                                     ctypes.byref(h)))
    return h.value


def moe_w4a16_forward_partial(h, hidden, topk_ids, topk_weights, partial, M, workspace, stream=None):
    _check(lib().moe_w4a16_forward_partial(h, _ptr(hidden), _ptr(topk_ids), _ptr(topk_weights),
                                           _ptr(partial), M, _ptr(workspace), workspace.numel(),
                                           _stream(stream)))


def moe_w4a16_finalize(acc, out, stream=None):
    _check(lib().moe_w4a16_finalize(_ptr(acc), _ptr(out), acc.numel(), _stream(stream)))


def moe_w4a16_destroy(h: int):
    _check(lib().moe_w4a16_destroy(h))


def moe_w4a16_pack(h, w1_q, w1_s, w2_q, w2_s, stream=None):
    _check(lib().moe_w4a16_pack(h, _ptr(w1_q), _ptr(w1_s), _ptr(w2_q), _ptr(w2_s), _stream(stream)))


def moe_w4a16_pack_ex(h, w1_q, w1_s, w2_q, w2_s, layout=LAYOUT_GPTQ, w1_g_idx=None, w2_g_idx=None,
                      stream=None):
    _check(lib().moe_w4a16_pack_ex(h, _ptr(w1_q), _ptr(w1_s), _ptr(w2_q), _ptr(w2_s), int(layout),
                                   _ptr(w1_g_idx), _ptr(w2_g_idx), _stream(stream)))


def moe_w4a16_workspace_size(h, M: int) -> int:
    return int(lib().moe_w4a16_workspace_size(h, M))


def moe_w4a16_host_staging_size(h, M: int) -> int:
    return int(lib().moe_w4a16_host_staging_size(h, M))


def moe_w4a16_forward(h, hidden, topk_ids, topk_weights, out, M, workspace, stream=None):
    _check(lib().moe_w4a16_forward(h, _ptr(hidden), _ptr(topk_ids), _ptr(topk_weights), _ptr(out),
                                   M, _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream(stream)))


def moe_w4a16_route(router_logits, M, E, topk, topk_ids, topk_weights, stream=None):
    _check(lib().moe_w4a16_route(_ptr(router_logits), M, E, topk, _ptr(topk_ids), _ptr(topk_weights),
                                 _stream(stream)))


def moe_w4a16_forward_logits(h, hidden, router_logits, topk_ids, topk_weights, out, M, workspace,
                             stream=None):
    _check(lib().moe_w4a16_forward_logits(h, _ptr(hidden), _ptr(router_logits), _ptr(topk_ids),
                                          _ptr(topk_weights), _ptr(out), M, _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_w4a16_forward_host(h, hidden, topk_ids, topk_weights, out, M, workspace, stream=None):
    _check(lib().moe_w4a16_forward_host(h, _ptr(hidden), _ptr(topk_ids), _ptr(topk_weights),
                                        _ptr(out), M, _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_w4a16_status(h, workspace, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check(lib().moe_w4a16_status(h, _ptr(workspace), ctypes.byref(v), _stream(stream)))
    return int(v.value)


def moe_w4a16_set_option(h, option: int, value: int):
    _check(lib().moe_w4a16_set_option(h, option, value))


def moe_w4a16_kernel_times(h, n: int = 5):
    buf = (ctypes.c_float * n)()
    w = lib().moe_w4a16_kernel_times(h, buf, n)
    if w < 0:
        _check(w)
    return [float(buf[i]) for i in range(w)]


def moe_w4a16_packed_bytes(h) -> int:
    return int(lib().moe_w4a16_packed_bytes(h))


def moe_w4a16_align_debug(topk_ids, M, topk, E, block, sorted_ids, expert_offsets, num_padded,
                          stream=None):
    _check(lib().moe_w4a16_align_debug(_ptr(topk_ids), M, topk, E, block, _ptr(sorted_ids),
                                       _ptr(expert_offsets), _ptr(num_padded), sorted_ids.numel(),
                                       _stream(stream)))


def moe_w4a16_unpack_debug(h, w1_q, w1_s, w2_q, w2_s, stream=None):
    _check(lib().moe_w4a16_unpack_debug(h, _ptr(w1_q), _ptr(w1_s), _ptr(w2_q), _ptr(w2_s),
                                        _stream(stream)))


def moe_w4a16_read_intermediate(h, workspace, M, h_rows, stream=None):
    _check(lib().moe_w4a16_read_intermediate(h, _ptr(workspace), M, _ptr(h_rows), _stream(stream)))


def moe_w4a16_read_accumulator(h, workspace, M, acc, stream=None):
    _check(lib().moe_w4a16_read_accumulator(h, _ptr(workspace), M, _ptr(acc), _stream(stream)))


def moe_w4a16_schedule_debug(h, workspace, M, n_ctas, stream=None):
    """Both GEMMs' stream-K boundaries of the last forward on ``workspace``:
    ``(bounds [2, n_ctas + 1] int64 list of lists, flags)``."""
    n = 2 * (n_ctas + 1)
    buf = (ctypes.c_int64 * n)()
    flags = _c_int(0)
    w = lib().moe_w4a16_schedule_debug(h, _ptr(workspace), M, buf, n, ctypes.byref(flags), _stream(stream))
    if w < 0:
        _check(w)
    vals = [int(buf[i]) for i in range(n)]
    return [vals[:n_ctas + 1], vals[n_ctas + 1:]], int(flags.value)


def moe_w4a16_forward_noalloc(h, hidden, topk_ids, topk_weights, out, M, stream=None):
    """The forward for callers that cannot allocate device memory: the workspace
    is a fixed array inside the library (see include/moe_w4a16.h)."""
    _check(lib().moe_w4a16_forward_noalloc(h, _ptr(hidden), _ptr(topk_ids), _ptr(topk_weights),
                                           _ptr(out), M, _stream(stream)))


class MoEW4A16:
    """Owns a library handle (packed weights) and a reusable device workspace."""

    def __init__(self, E: int, K: int, N: int, topk: int, group_size: int = 32, expert_range=None):
        """``E`` experts of hidden size ``K`` and intermediate size ``N``; with
        ``expert_range=(begin, end)`` the handle holds only experts [begin, end) of
        the ``E`` (expert parallelism: pack takes those experts' weights)."""
        self.E_total = E
        self.K, self.N, self.topk = K, N, topk
        if expert_range is None:
            self.expert_begin, self.E = 0, E
            self.handle = moe_w4a16_create(E, K, N, topk, group_size)
        else:
            b, e = (int(v) for v in expert_range)
            self.expert_begin, self.E = b, e - b
            self.handle = moe_w4a16_create_ep(E, b, e, K, N, topk, group_size)
        self.workspace = None

    def close(self):
        if self.handle:
            moe_w4a16_destroy(self.handle)
            self.handle = None
            self.workspace = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def pack(self, w1_q, w1_s, w2_q, w2_s, stream=None, layout=LAYOUT_GPTQ, w1_g_idx=None,
             w2_g_idx=None):
        """Repack the weights; ``layout`` GPTQ (codes [E, R/8, C]) or compressed-tensors
        (codes [E, C, R/8]); optional act-order group indices [E, K] / [E, N]."""
        E, K, N = self.E, self.K, self.N
        if layout == LAYOUT_GPTQ:
            shapes = [(E, K // 8, 2 * N), (E, K // 32, 2 * N), (E, N // 8, K), (E, N // 32, K)]
        else:
            shapes = [(E, 2 * N, K // 8), (E, 2 * N, K // 32), (E, K, N // 8), (E, K, N // 32)]
        _need(w1_q, ("int32",), shapes[0], "w1_q")
        _need(w1_s, _BITS16, shapes[1], "w1_s")
        _need(w2_q, ("int32",), shapes[2], "w2_q")
        _need(w2_s, _BITS16, shapes[3], "w2_s")
        if w1_g_idx is not None:
            _need(w1_g_idx, ("int32",), (E, K), "w1_g_idx")
        if w2_g_idx is not None:
            _need(w2_g_idx, ("int32",), (E, N), "w2_g_idx")
        if layout == LAYOUT_GPTQ and w1_g_idx is None and w2_g_idx is None:
            moe_w4a16_pack(self.handle, w1_q, w1_s, w2_q, w2_s, stream)
        else:
            moe_w4a16_pack_ex(self.handle, w1_q, w1_s, w2_q, w2_s, layout, w1_g_idx, w2_g_idx, stream)

    def ensure_workspace(self, M: int, host_staging: bool = False):
        # (asked every call: the size depends on the handle's options, which the
        # caller may change between calls)
        need = moe_w4a16_workspace_size(self.handle, M)
        if host_staging:
            need += moe_w4a16_host_staging_size(self.handle, M)
        if self.workspace is None or self.workspace.numel() < need:
            import torch
            self.workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
        return self.workspace

    def forward(self, hidden, topk_ids, topk_weights, out=None, stream=None):
        import torch
        M = hidden.shape[0]
        _need(hidden, _BITS16, (M, self.K), "hidden")
        _need(topk_ids, ("int32",), (M, self.topk), "topk_ids")
        _need(topk_weights, ("float32",), (M, self.topk), "topk_weights")
        if out is None:
            out = torch.empty((M, self.K), dtype=torch.bfloat16, device=hidden.device)
        _need(out, _BITS16, (M, self.K), "out")
        ws = self.ensure_workspace(M)
        moe_w4a16_forward(self.handle, hidden, topk_ids, topk_weights, out, M, ws, stream)
        return out

    def forward_partial(self, hidden, topk_ids, topk_weights, partial=None, stream=None):
        """fp32 [M, K] weighted sum over this handle's experts (no bf16 rounding)."""
        import torch
        M = hidden.shape[0]
        _need(hidden, _BITS16, (M, self.K), "hidden")
        _need(topk_ids, ("int32",), (M, self.topk), "topk_ids")
        _need(topk_weights, ("float32",), (M, self.topk), "topk_weights")
        if partial is None:
            partial = torch.empty((M, self.K), dtype=torch.float32, device=hidden.device)
        _need(partial, ("float32",), (M, self.K), "partial")
        ws = self.ensure_workspace(M)
        moe_w4a16_forward_partial(self.handle, hidden, topk_ids, topk_weights, partial, M, ws, stream)
        return partial

    def route(self, router_logits, stream=None):
        """Top-k routing of ``router_logits`` fp32 [M, E] on the device: (ids, weights)."""
        import torch
        M = router_logits.shape[0]
        _need(router_logits, ("float32",), (M, self.E_total), "router_logits")
        ids = torch.empty((M, self.topk), dtype=torch.int32, device=router_logits.device)
        w = torch.empty((M, self.topk), dtype=torch.float32, device=router_logits.device)
        moe_w4a16_route(router_logits, M, self.E_total, self.topk, ids, w, stream)
        return ids, w

    def forward_logits(self, hidden, router_logits, out=None, stream=None):
        """Routing plus forward: (out, topk_ids, topk_weights)."""
        import torch
        M = hidden.shape[0]
        _need(hidden, _BITS16, (M, self.K), "hidden")
        _need(router_logits, ("float32",), (M, self.E_total), "router_logits")
        if out is None:
            out = torch.empty((M, self.K), dtype=torch.bfloat16, device=hidden.device)
        _need(out, _BITS16, (M, self.K), "out")
        ids = torch.empty((M, self.topk), dtype=torch.int32, device=hidden.device)
        w = torch.empty((M, self.topk), dtype=torch.float32, device=hidden.device)
        ws = self.ensure_workspace(M)
        moe_w4a16_forward_logits(self.handle, hidden, router_logits, ids, w, out, M, ws, stream)
        return out, ids, w

    def forward_host(self, hidden, topk_ids, topk_weights, out, stream=None):
        M = hidden.shape[0]
        _need(hidden, _BITS16, (M, self.K), "hidden", device=False)
        _need(topk_ids, ("int32",), (M, self.topk), "topk_ids", device=False)
        _need(topk_weights, ("float32",), (M, self.topk), "topk_weights", device=False)
        _need(out, _BITS16, (M, self.K), "out", device=False)
        ws = self.ensure_workspace(M, host_staging=True)
        moe_w4a16_forward_host(self.handle, hidden, topk_ids, topk_weights, out, M, ws, stream)
        return out

    def status(self, stream=None) -> int:
        return moe_w4a16_status(self.handle, self.workspace, stream)

    def accumulator(self, M: int, stream=None):
        """fp32 [M, K] output accumulator of the last forward (before the bf16 rounding)."""
        import torch
        acc = torch.zeros((M, self.K), dtype=torch.float32, device="cuda")
        moe_w4a16_read_accumulator(self.handle, self.workspace, M, acc, stream)
        return acc

    def intermediate(self, M: int, stream=None):
        import torch
        h_rows = torch.zeros((M * self.topk, self.N), dtype=torch.float32, device="cuda")
        moe_w4a16_read_intermediate(self.handle, self.workspace, M, h_rows, stream)
        return h_rows
