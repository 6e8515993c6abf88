"""Data-parallel sharding of the forward over ranks (host logic only).

The differential-attention forward is independent across (batch, head)
units (V1) and (batch, KV group) units (V2): no step of the path exchanges
data between units, so ranks split the batch and need no collective on the
data path.  Under weak scaling every rank owns ``per_rank`` whole batch
entries; the global batch is ``per_rank * world``.
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
