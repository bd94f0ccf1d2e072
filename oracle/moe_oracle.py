"""CPU oracle for the INT4 weight-only (W4A16) fused Mixture-of-Experts feed-forward.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or run
this module: only the tests, the smoke check and the benchmark's CPU-baseline
leg use it. It shares no code with the CUDA library; the two meet only in the
seeded inputs of ``int4_weight_only_moe_gb300.inputs``.

Everything is plain numpy in float64, slow and written to be checked by eye
against the definitions it follows:

* Weight format -- "The Pivot to Real Hardware: ... INT4 MoE Benchmark for Kimi
  K2.6", Step 1 (Understanding the Weight Format) and Input Knowledge item 2:
  INT4 values are packed eight per int32 in the logical GPTQ format; w1 fuses the
  gate and up projections of a SwiGLU MLP (2N outputs), w2 is the down
  projection; each group of 32 values along the reduction dimension shares one
  scale (group_size=32, also "The Commit That Captured a Plateau", commit text).
* Symmetric code: a stored nibble ``u`` in ``0..15`` stands for ``u - 8``.
* Expert MLP: ``down(SiLU(gate . x) * (up . x))`` with ``SiLU(z) = z / (1 + e^-z)``.
* Mixture: every token is routed to its top-k experts and the k expert outputs
  are summed with the top-k weights (Input Knowledge item 1: 384 experts, top-8).
* Routing (the gating network that chooses which experts a token is sent to --
  "The Weight-Streaming Threshold", Input Knowledge Required; the workloads'
  recipe "router logits -> softmax top-k, renormalised"): softmax over all E
  router logits of a token, keep the k most probable experts, divide their
  probabilities by their sum. Equal logits rank the lower expert id first.
* Align (the token->expert counting sort that groups routed rows by expert and
  pads every expert's rows to a block size) -- the pages only mention "sorting
  indices"; the definition used here is the plainest one: experts in id order,
  inside an expert the flat slot ids ``t*k + j`` in ascending order, every
  expert's row count rounded up to a multiple of ``block`` with the sentinel
  ``M*k``, experts with no rows get none.

Readings where the pages are silent (each also listed in the design notes):
nibble ``i`` of a word holds element ``8*row + i`` (lowest bits first); gate
rows are ``[0, N)`` and up rows ``[N, 2N)`` of w1; w2's groups run along its own
reduction dimension N; scales are bf16.

Pins: every function here is checked in ``tests/test_oracle_pins.py`` against
hand-derived golden values, brute force on tiny inputs, library routines in
special cases and algebraic invariants -- none of which re-type these formulas.
"""
from __future__ import annotations

import numpy as np

GROUP_SIZE = 32


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (a bf16 is the top half of a float32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def unpack_codes(qweight: np.ndarray) -> np.ndarray:
    """Stored 4-bit codes ``u`` of a packed ``[R/8, C]`` int32 matrix -> ``[R, C]`` int64.

    Code ``i`` of word ``[r, c]`` sits in bits ``4i..4i+3`` and is element
    ``(8r + i, c)`` (eight INT4 values per int32 along the reduction axis).
    """
    q = np.asarray(qweight).view(np.uint32).astype(np.int64)
    r8, c = q.shape
    u = np.empty((r8 * 8, c), dtype=np.int64)
    for i in range(8):
        u[i::8, :] = (q >> (4 * i)) & 0xF
    return u


def dequantize(qweight: np.ndarray, scales: np.ndarray, group_size: int = GROUP_SIZE) -> np.ndarray:
    """Dequantised weight ``[C, R]`` (output-feature major) of a packed ``[R/8, C]`` matrix.

    ``W[c, r] = (u[r, c] - 8) * scale[r // group_size, c]`` -- symmetric INT4, one
    bf16 scale per group of ``group_size`` reduction elements.
    """
    u = unpack_codes(qweight)                       # [R, C]
    s = bf16_to_f64(scales)                         # [R/G, C]
    s_full = np.repeat(s, group_size, axis=0)       # [R, C]
    return ((u - 8).astype(np.float64) * s_full).T  # [C, R]


def unpack_codes_ct(weight_packed: np.ndarray) -> np.ndarray:
    """Stored 4-bit codes of a compressed-tensors packed ``[C, R/8]`` int32 matrix -> ``[R, C]`` int64.

    The compressed-tensors INT4 layout ("The Pivot to Real Hardware ...", The
    Context: Where We Stand -- the model ships in that format) keeps every output
    feature's row contiguous: word ``[c, r]`` holds elements ``(8r + i, c)`` of
    the reduction axis, code ``i`` in bits ``4i..4i+3`` (lowest first), with the
    same symmetric offset (a code ``u`` stands for ``u - 8``).
    """
    q = np.asarray(weight_packed).view(np.uint32).astype(np.int64)
    c, r8 = q.shape
    u = np.empty((r8 * 8, c), dtype=np.int64)
    for i in range(8):
        u[i::8, :] = ((q >> (4 * i)) & 0xF).T
    return u


def dequantize_ct(weight_packed: np.ndarray, weight_scale: np.ndarray,
                  group_size: int = GROUP_SIZE) -> np.ndarray:
    """Dequantised weight ``[C, R]`` of a compressed-tensors matrix.

    ``W[c, r] = (u[r, c] - 8) * scale[c, r // group_size]`` with the codes of
    ``unpack_codes_ct`` and the scales stored feature-major, ``[C, R/G]`` bf16.
    """
    u = unpack_codes_ct(weight_packed)                       # [R, C]
    s = bf16_to_f64(weight_scale)                            # [C, R/G]
    s_full = np.repeat(s, group_size, axis=1)                # [C, R]
    return (u.T - 8).astype(np.float64) * s_full             # [C, R]


def dequantize_g_idx(qweight: np.ndarray, scales: np.ndarray, g_idx: np.ndarray) -> np.ndarray:
    """Dequantised weight ``[C, R]`` of a GPTQ matrix quantised in activation order.

    With act-order ("The Pivot to Real Hardware ...", Step 2: the repack's
    permutation and group-index tensors) reduction element ``r`` belongs to the
    scale group ``g_idx[r]`` instead of ``r // 32``:
    ``W[c, r] = (u[r, c] - 8) * scale[g_idx[r], c]``. The codes stay in the
    natural order of ``r``.
    """
    u = unpack_codes(qweight)                                # [R, C]
    s = bf16_to_f64(scales)                                  # [R/G, C]
    g = np.asarray(g_idx, dtype=np.int64)
    return ((u - 8).astype(np.float64) * s[g, :]).T          # [C, R]


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU (swish): ``z * sigmoid(z) = z / (1 + exp(-z))``."""
    return z / (1.0 + np.exp(-z))


def expert_hidden(x: np.ndarray, w1: np.ndarray) -> np.ndarray:
    """Intermediate activations ``h = SiLU(x W1[:N]^T) * (x W1[N:]^T)``, ``[T, N]``.

    ``w1 [2N, K]`` holds the gate rows first and the up rows second.
    """
    n = w1.shape[0] // 2
    gate = x @ w1[:n].T
    up = x @ w1[n:].T
    return silu(gate) * up


def expert_ffn(x: np.ndarray, w1: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """SwiGLU expert MLP on rows ``x [T, K]`` with dense ``w1 [2N, K]``, ``w2 [K, N]``.

    ``gate = x W1[:N]^T``, ``up = x W1[N:]^T``, ``h = SiLU(gate) * up``, ``y = h W2^T``.
    """
    return expert_hidden(x, w1) @ w2.T


def expert_dense(w1_q, w1_s, w2_q, w2_s, e: int, group_size: int = GROUP_SIZE):
    """Dense float64 ``(W1 [2N, K], W2 [K, N])`` of expert ``e`` from the packed inputs."""
    return (dequantize(w1_q[e], w1_s[e], group_size),
            dequantize(w2_q[e], w2_s[e], group_size))


def moe_forward(hidden_bf16, topk_ids, topk_weights, w1_q, w1_s, w2_q, w2_s,
                tokens=None, group_size: int = GROUP_SIZE, expert_source=None,
                dense_source=None) -> np.ndarray:
    """Fused MoE feed-forward, float64 ``[len(tokens), K]``.

    ``out[t] = sum_j topk_weights[t, j] * FFN_{topk_ids[t, j]}(x_t)``.

    ``tokens`` restricts the computation to those rows (a sampled check of a
    large batch). ``expert_source(e)`` may supply ``(w1_q, w1_s, w2_q, w2_s)`` of
    one expert instead of indexing the stacked arrays (so that a caller can
    regenerate only the experts it needs); ``dense_source(e)`` may instead
    supply expert ``e``'s dequantised ``(W1 [2N, K], W2 [K, N])`` (weights held in
    another packed layout). Slot ids outside ``[0, E)`` are skipped. Experts are
    visited one at a time, each dequantised once.
    """
    x_all = bf16_to_f64(hidden_bf16)
    ids = np.asarray(topk_ids)
    wts = np.asarray(topk_weights, dtype=np.float64)
    M, k = ids.shape
    rows = np.arange(M) if tokens is None else np.asarray(tokens)
    K = x_all.shape[1]
    out = np.zeros((len(rows), K), dtype=np.float64)
    sub_ids = ids[rows]
    if expert_source is None and dense_source is None:
        E = w1_q.shape[0]
    else:
        E = None
    for e in np.unique(sub_ids):
        if e < 0 or (E is not None and e >= E):
            continue
        if dense_source is not None:
            w1, w2 = dense_source(int(e))
        elif expert_source is None:
            w1, w2 = expert_dense(w1_q, w1_s, w2_q, w2_s, int(e), group_size)
        else:
            q1, s1, q2, s2 = expert_source(int(e))
            w1, w2 = dequantize(q1, s1, group_size), dequantize(q2, s2, group_size)
        r_idx, j_idx = np.nonzero(sub_ids == e)
        y = expert_ffn(x_all[rows[r_idx]], w1, w2)          # [n_e, K]
        y *= wts[rows[r_idx], j_idx][:, None]
        np.add.at(out, r_idx, y)
    return out


def route(logits: np.ndarray, topk: int):
    """Top-k routing of router logits ``[M, E]``: ``(topk_ids int32 [M, k], topk_weights float64 [M, k])``.

    For every token: ``p = softmax(logits)`` over all ``E`` experts; the ids are
    the ``k`` experts of largest ``p`` (equivalently largest logit) in descending
    order, equal logits taken in ascending expert id; the weights are those
    ``p`` divided by their sum (renormalised to 1).
    """
    lg = np.asarray(logits, dtype=np.float64)
    M, E = lg.shape
    ids = np.empty((M, topk), dtype=np.int32)
    wts = np.empty((M, topk), dtype=np.float64)
    for t in range(M):
        row = lg[t]
        p = np.exp(row - row.max())
        p /= p.sum()
        order = sorted(range(E), key=lambda e: (-row[e], e))[:topk]
        sel = p[order]
        ids[t] = order
        wts[t] = sel / sel.sum()
    return ids, wts


def moe_align(topk_ids: np.ndarray, num_experts: int, block: int):
    """Token->expert counting sort with per-expert padding to ``block`` rows.

    Returns ``(sorted_ids, expert_offsets, num_padded)``:

    * ``sorted_ids`` int32 ``[num_padded]`` -- for each expert ``e`` in id order,
      the flat slot ids ``t*k + j`` with ``topk_ids[t, j] == e`` in ascending
      order, then the sentinel ``M*k`` up to the next multiple of ``block``;
    * ``expert_offsets`` int32 ``[E + 1]`` -- start of every expert's segment;
    * ``num_padded`` -- total length.

    Slot ids outside ``[0, E)`` are left out.
    """
    flat = np.asarray(topk_ids).reshape(-1).astype(np.int64)
    sentinel = flat.size
    valid = (flat >= 0) & (flat < num_experts)
    counts = np.bincount(flat[valid], minlength=num_experts)
    padded = -(-counts // block) * block
    offsets = np.zeros(num_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(padded)
    order = np.nonzero(valid)[0]
    order = order[np.argsort(flat[order], kind="stable")]
    sorted_ids = np.full(int(offsets[-1]), sentinel, dtype=np.int64)
    start = 0
    for e in range(num_experts):
        c = int(counts[e])
        sorted_ids[offsets[e]:offsets[e] + c] = order[start:start + c]
        start += c
    return sorted_ids.astype(np.int32), offsets.astype(np.int32), int(offsets[-1])


def roofline_bytes_per_expert(K: int, N: int, group_size: int = GROUP_SIZE) -> int:
    """Packed INT4 weight plus bf16 scale bytes of one expert (w1 gate+up and w2)."""
    w = (2 * N * K + K * N) // 2
    s = (2 * N * (K // group_size) + K * (N // group_size)) * 2
    return w + s
