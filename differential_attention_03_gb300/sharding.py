"""Data-parallel sharding over ranks (host logic only).

The differential-attention forward is independent across (batch, head)
units (V1) and (batch, KV group) units (V2): no step of the path exchanges
data between units, so ranks split the batch and need no collective on the
data path.  Under weak scaling every rank owns ``per_rank`` whole batch
entries; the global batch is ``per_rank * world``.  The backward adds one
exchange: the gradients of the parameters every rank shares (lambda, gamma,
logits shared by all sequences) are summed over the ranks
(``allreduce_shared_grads``).
"""

from __future__ import annotations


def batch_slice(global_batch: int, world: int, rank: int) -> tuple[int, int]:
    """[start, stop) of the batch entries rank ``rank`` owns (contiguous, balanced)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    base, extra = divmod(global_batch, world)
    start = rank * base + min(rank, extra)
    stop = start + base + (1 if rank < extra else 0)
    return start, stop


def weak_scaling_seed(seed: int, rank: int) -> int:
    """Seed of rank ``rank``'s own synthetic batch under weak scaling."""
    return seed + 1000 * rank


def allreduce_shared_grads(grads, group=None):
    """Sum, over the data-parallel ranks, the gradients of parameters all ranks share.

    The backward's only exchange step: dq, dk and dv belong to each rank's own
    batch entries, but lambda (or its four vectors), gamma and V2 logits shared
    by every sequence receive a share of their gradient from every rank's
    entries.  ``grads`` is a list of tensors on one device (CUDA tensors with
    the NCCL backend, CPU tensors with gloo), summed in place with one
    all_reduce over a flat buffer.
    """
    import torch
    import torch.distributed as dist

    if not grads:
        return grads
    if len({(g.dtype, g.device) for g in grads}) != 1:
        raise ValueError("shared gradients must have one dtype and one device (no silent down-casts)")
    flat = torch.cat([g.reshape(-1) for g in grads])
    dist.all_reduce(flat, op=dist.ReduceOp.SUM, group=group)
    off = 0
    for g in grads:
        n = g.numel()
        g.copy_(flat[off:off + n].view_as(g))
        off += n
    return grads
