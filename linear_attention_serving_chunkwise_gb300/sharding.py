"""Partition KDA work across ranks (one process per GPU).

Sequences and heads never exchange data, so N GPUs take N disjoint sets of
(sequence, head) units and need no collective on the data path.  These helpers
decide who takes what; they hold no KDA arithmetic.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple


def shard_heads(num_heads: int, world: int, rank: int) -> Tuple[int, int]:
    """Contiguous head range [h0, h1) of `rank`; sizes differ by at most one."""
    if not (0 <= rank < world) or num_heads < 0:
        raise ValueError("bad rank/world/num_heads")
    base, extra = divmod(num_heads, world)
    h0 = rank * base + min(rank, extra)
    return h0, h0 + base + (1 if rank < extra else 0)


def shard_sequences(seqlens: Sequence[int], world: int, rank: int) -> List[int]:
    """Indices of the sequences `rank` takes, balancing tokens: longest first, each
    to the currently lightest rank (ties to the lower rank).  Deterministic."""
    if not (0 <= rank < world):
        raise ValueError("bad rank/world")
    order = sorted(range(len(seqlens)), key=lambda i: (-int(seqlens[i]), i))
    load = [0] * world
    owner = {}
    for i in order:
        r = min(range(world), key=lambda x: (load[x], x))
        owner[i] = r
        load[r] += int(seqlens[i])
    return sorted(i for i in owner if owner[i] == rank)
