"""Expert parallelism over ranks ("The Weight-Streaming Threshold", Assumptions
Embedded in the Analysis: each GPU of a TP-8 group holds a subset of the experts
and an AllReduce combines their outputs).

Rank r of G holds a contiguous range of the layer's experts (``expert_range``);
its forward is the fp32 partial sum over those experts
(``MoEW4A16.forward_partial``); one sum-reduce over the ranks
(``torch.distributed.all_reduce``, NCCL between GPUs, gloo on the host) adds the
partials, and ``finalize`` rounds the sum to bf16 on the device. The only
exchange is that reduce: routing is replicated (every rank sees every token's
ids) and no activations move between ranks.
"""
from __future__ import annotations


def expert_range(E: int, world: int, rank: int):
    """Experts ``[begin, end)`` of rank ``rank`` when ``E`` experts are split into
    ``world`` contiguous ranges whose sizes differ by at most one (the first
    ``E % world`` ranks take one more)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need world >= 1 and 0 <= rank < world")
    if E < world:
        raise ValueError("every rank needs at least one expert")
    base, extra = divmod(E, world)
    begin = rank * base + min(rank, extra)
    return begin, begin + base + (1 if rank < extra else 0)


def allreduce_partial(partial, group=None):
    """Sum the ranks' fp32 partials in place (one collective) and return it."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(partial, op=dist.ReduceOp.SUM, group=group)
    return partial


def finalize(acc, out=None, stream=None):
    """bf16 round-to-nearest-even of an fp32 [M, K] sum, on the device."""
    import torch
    from . import moe_w4a16_finalize
    if out is None:
        out = torch.empty(acc.shape, dtype=torch.bfloat16, device=acc.device)
    moe_w4a16_finalize(acc, out, stream)
    return out


def ep_forward(moe, hidden, topk_ids, topk_weights, group=None, stream=None):
    """One expert-parallel forward: this rank's partial, the sum-reduce, the rounding."""
    partial = moe.forward_partial(hidden, topk_ids, topk_weights, stream=stream)
    allreduce_partial(partial, group)
    return finalize(partial, stream=stream)
