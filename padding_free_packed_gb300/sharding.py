"""Splitting one packed batch across data-parallel ranks.

Sequences never attend across cu_seqlens boundaries (page "Source code for
gigl.nn.packed_attention", module docstring: each sequence attends only to
itself), so a batch shards by sequence with no collective on the attention
path: each rank packs and runs its own subset. Attention costs L_i^2 per
sequence, so sequences are assigned longest-processing-time first to the
rank with the least accumulated cost. Host logic only; it launches nothing.
"""

from __future__ import annotations

import heapq

import numpy as np


def shard_sequences(lengths, world_size: int) -> list[np.ndarray]:
    """Returns, per rank, the ascending indices of the sequences it owns.

    Greedy longest-first assignment on cost L_i^2 (ties broken by sequence
    index, then rank index, so every rank computes the same partition).
    """
    if world_size < 1:
        raise ValueError("world_size must be >= 1")
    lengths = np.asarray(lengths, dtype=np.int64)
    order = sorted(range(lengths.shape[0]), key=lambda i: (-int(lengths[i]), i))
    heap = [(0, r) for r in range(world_size)]
    owned: list[list[int]] = [[] for _ in range(world_size)]
    for i in order:
        cost, r = heapq.heappop(heap)
        owned[r].append(i)
        heapq.heappush(heap, (cost + int(lengths[i]) ** 2, r))
    return [np.array(sorted(o), dtype=np.int64) for o in owned]


def shard_cost(lengths, shards) -> list[int]:
    """Attention cost (sum of L_i^2) of each rank's shard."""
    lengths = np.asarray(lengths, dtype=np.int64)
    return [int((lengths[s] ** 2).sum()) for s in shards]
