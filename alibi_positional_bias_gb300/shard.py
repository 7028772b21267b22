"""Sharding of the attention work across ranks.

Every (b, h) pair of the ALiBi attention path is an independent problem (the
bias depends only on the head's slope and the positions inside the sequence),
so a global batch splits across ranks with no exchange step: each rank runs
its contiguous range of sequences through the same kernels. Only the host
decides the ranges; nothing here touches device memory.
"""
from __future__ import annotations


def shard_range(units: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous [start, start + count) share of ``units`` for ``rank`` of ``world``.

    The first ``units % world`` ranks get one extra unit; counts differ by at most one.
    """
    if world < 1 or not (0 <= rank < world) or units < 0:
        raise ValueError("need world >= 1, 0 <= rank < world, units >= 0")
    base, extra = divmod(units, world)
    start = rank * base + min(rank, extra)
    return start, base + (1 if rank < extra else 0)


def shard_batch(B: int, world: int, rank: int) -> tuple[int, int]:
    """Sequences [b0, b0 + nb) of a global batch of B handled by ``rank``.

    Sharding by whole sequences keeps all H heads of a sequence on one rank, so
    each rank's tensors are a contiguous slice of the global [B, H, N, d] ones.
    """
    return shard_range(B, world, rank)
