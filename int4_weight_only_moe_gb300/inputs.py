"""Seeded synthetic inputs for the W4A16 fused Mixture-of-Experts feed-forward.

This module draws random numbers and lays them out in the input formats of the
two library calls; it holds none of the method's arithmetic (no dequantisation,
no matmul, no activation, no routing-weighted sum). Both the CUDA path and the
CPU oracle take their inputs from here, so the two sides see identical bytes.

Formats produced (the GPTQ-style "logical" input format that the repack step of
"The Pivot to Real Hardware ..." (Step 1 and Step 2) starts from):

* ``w1_q``  int32 ``[E, K/8, 2N]``: gate rows ``[0, N)`` then up rows ``[N, 2N)``
  along the last axis; eight 4-bit codes per word along the reduction axis K,
  code ``i`` of word ``[e, r, c]`` in bits ``4i..4i+3`` is element ``8r+i``.
* ``w1_s``  uint16 (bf16 bit patterns) ``[E, K/32, 2N]``: one scale per group of
  32 consecutive reduction elements.
* ``w2_q``  int32 ``[E, N/8, K]`` and ``w2_s`` uint16 ``[E, N/32, K]``: the down
  projection, reduction axis N.
* ``hidden`` uint16 (bf16) ``[M, K]``; router ``logits`` float32 ``[M, E]``.
  (Turning logits into ``topk_ids`` / ``topk_weights`` is the router, a step of
  the method: the library's router kernel does it on the device, the oracle's
  ``route`` on the host; nothing here does.)

Every random 32-bit word is uniform, so all eight codes of a word are uniform
on ``0..15`` (stored value ``u``; the symmetric code is ``u - 8`` in ``[-8, 7]``).
Scales are uniform on ``[0.005, 0.02]`` rounded to bf16, hidden states are
standard normal rounded to bf16, and router logits follow the workload recipe
(normal, uniform, or Zipf-skewed expert popularity with Gumbel noise), rounded to
float32.

Expert weights are drawn from a per-expert stream, so a caller that needs only
a few experts (a sampled oracle check at full size) regenerates just those.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

WEIGHT_SEED = 0
HIDDEN_SEED = 1
ROUTING_SEED = 2
GROUP_SIZE = 32


@dataclass(frozen=True)
class Workload:
    """Shape and input recipe of one benchmark/parity workload."""

    name: str
    E: int
    K: int
    N: int
    topk: int
    M: int
    routing: str  # "normal" | "uniform" | "zipf"
    zipf_s: float = 1.1
    note: str = field(default="", compare=False)


# The workloads at the dimensions of the benchmark described on the pages
# (Kimi K2.6 MoE layer: 384 experts, hidden 7168, intermediate 2048, top-8,
# INT4 symmetric group 32) plus a tiny case small enough for exhaustive checks.
WORKLOADS = {
    "tiny": Workload("tiny", 8, 256, 128, 2, 4, "normal"),
    "decode": Workload("decode", 384, 7168, 2048, 8, 1, "uniform"),
    "small9": Workload("small9", 384, 7168, 2048, 8, 9, "normal"),
    "small32": Workload("small32", 384, 7168, 2048, 8, 32, "normal"),
    "small90": Workload("small90", 384, 7168, 2048, 8, 90, "normal"),
    "plateau256": Workload("plateau256", 384, 7168, 2048, 8, 256, "normal"),
    "plateau512": Workload("plateau512", 384, 7168, 2048, 8, 512, "normal"),
    "large_uniform": Workload("large_uniform", 384, 7168, 2048, 8, 1024, "uniform"),
    "large_zipf": Workload("large_zipf", 384, 7168, 2048, 8, 1024, "zipf"),
}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); return the bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(list(key)))


def expert_weights(e: int, K: int, N: int, seed: int = WEIGHT_SEED):
    """Random GPTQ-style packed weights and bf16 scales of expert ``e``.

    Returns ``(w1_q [K/8, 2N] int32, w1_s [K/32, 2N] uint16,
    w2_q [N/8, K] int32, w2_s [N/32, K] uint16)``.
    """
    g = _rng(seed, 1000 + e)
    w1_q = g.integers(0, 2**32, size=(K // 8, 2 * N), dtype=np.uint32).view(np.int32)
    w1_s = f32_to_bf16_bits(g.uniform(0.005, 0.02, size=(K // GROUP_SIZE, 2 * N)))
    w2_q = g.integers(0, 2**32, size=(N // 8, K), dtype=np.uint32).view(np.int32)
    w2_s = f32_to_bf16_bits(g.uniform(0.005, 0.02, size=(N // GROUP_SIZE, K)))
    return w1_q, w1_s, w2_q, w2_s


def all_expert_weights(E: int, K: int, N: int, seed: int = WEIGHT_SEED):
    """Stack :func:`expert_weights` over ``E`` experts (host memory)."""
    w1_q = np.empty((E, K // 8, 2 * N), np.int32)
    w1_s = np.empty((E, K // GROUP_SIZE, 2 * N), np.uint16)
    w2_q = np.empty((E, N // 8, K), np.int32)
    w2_s = np.empty((E, N // GROUP_SIZE, K), np.uint16)
    for e in range(E):
        w1_q[e], w1_s[e], w2_q[e], w2_s[e] = expert_weights(e, K, N, seed)
    return w1_q, w1_s, w2_q, w2_s


def expert_weights_ct(e: int, K: int, N: int, seed: int = WEIGHT_SEED):
    """Random weights of expert ``e`` in the compressed-tensors packed layout.

    Every output feature's reduction row is contiguous: returns
    ``(w1_q [2N, K/8] int32, w1_s [2N, K/32] uint16, w2_q [K, N/8] int32,
    w2_s [K, N/32] uint16)``; code ``i`` of word ``[c, r]`` in bits ``4i..4i+3``
    is reduction element ``8r+i`` of feature ``c``.
    """
    g = _rng(seed, 3000 + e)
    w1_q = g.integers(0, 2**32, size=(2 * N, K // 8), dtype=np.uint32).view(np.int32)
    w1_s = f32_to_bf16_bits(g.uniform(0.005, 0.02, size=(2 * N, K // GROUP_SIZE)))
    w2_q = g.integers(0, 2**32, size=(K, N // 8), dtype=np.uint32).view(np.int32)
    w2_s = f32_to_bf16_bits(g.uniform(0.005, 0.02, size=(K, N // GROUP_SIZE)))
    return w1_q, w1_s, w2_q, w2_s


def act_order_g_idx(e: int, R: int, which: int, seed: int = WEIGHT_SEED) -> np.ndarray:
    """Group index ``[R]`` int32 of a matrix quantised in a random activation order.

    A seeded random order of the ``R`` reduction channels is cut into runs of 32;
    channel ``c`` gets the number of the run it falls in, so every group has
    exactly 32 members, scattered over the axis. ``which`` tells w1 (0) from
    w2 (1).
    """
    order = _rng(seed, 5000 + e, which).permutation(R)
    g_idx = np.empty(R, dtype=np.int32)
    g_idx[order] = np.arange(R, dtype=np.int32) // GROUP_SIZE
    return g_idx


def hidden_states(M: int, K: int, seed: int = HIDDEN_SEED, step: int = 0) -> np.ndarray:
    """bf16 bit patterns of ``M`` standard-normal hidden vectors of length ``K``."""
    g = _rng(seed, 7, step)
    return f32_to_bf16_bits(g.standard_normal((M, K), dtype=np.float32))


def router_logits(M: int, E: int, routing: str, seed: int = ROUTING_SEED,
                  step: int = 0, zipf_s: float = 1.1) -> np.ndarray:
    """Router logits ``[M, E]`` (float32) following the workload's recipe."""
    return _router_logits64(M, E, routing, seed, step, zipf_s).astype(np.float32)


def _router_logits64(M, E, routing, seed, step, zipf_s):
    g = _rng(seed, 11, step)
    if routing == "normal":
        return g.standard_normal((M, E))
    if routing == "uniform":
        return g.uniform(0.0, 1.0, size=(M, E))
    if routing == "zipf":
        # expert popularity p ~ rank^-s over a seeded random rank->expert map;
        # adding Gumbel noise to log p makes top-k a draw without replacement
        # proportional to p.
        perm = _rng(seed, 13).permutation(E)
        p = np.empty(E)
        p[perm] = np.arange(1, E + 1, dtype=np.float64) ** (-zipf_s)
        p /= p.sum()
        return np.log(p)[None, :] + g.gumbel(size=(M, E))
    raise ValueError(f"unknown routing recipe {routing!r}")


def workload_inputs(wl: Workload, step: int = 0, M: int | None = None):
    """Activations and router logits of one step of ``wl``: (hidden bf16 bits, logits float32)."""
    m = wl.M if M is None else M
    return hidden_states(m, wl.K, step=step), router_logits(m, wl.E, wl.routing, step=step, zipf_s=wl.zipf_s)


def active_experts(topk_ids: np.ndarray) -> np.ndarray:
    """Sorted unique expert ids referenced by a routing tensor."""
    return np.unique(np.asarray(topk_ids).reshape(-1))
