"""Data-parallel sharding of a packed batch, checked with two gloo ranks on CPU.

Every rank computes the partition independently; the ranks then all-gather
their shards and check that together they cover every sequence exactly once,
that they agree with each other, and that the longest-first assignment keeps
the attention cost (sum of L^2) balanced.
"""

import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from padding_free_packed_gb300 import workloads
from padding_free_packed_gb300.sharding import shard_cost, shard_sequences


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        for name in ("graph_fp32", "contrastive_bf16", "longdoc_bf16"):
            lengths = workloads.draw_lengths(name, np.random.default_rng(0))
            shards = shard_sequences(lengths, world)
            mine = torch.from_numpy(shards[rank])
            sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
            dist.all_gather(sizes, torch.tensor([mine.numel()]))
            width = max(int(s.item()) for s in sizes)
            padded = torch.full((width,), -1, dtype=torch.int64)
            padded[: mine.numel()] = mine
            gathered = [torch.zeros(width, dtype=torch.int64) for _ in range(world)]
            dist.all_gather(gathered, padded)
            gathered = [g[: int(n.item())] for g, n in zip(gathered, sizes)]
            allidx = torch.cat(gathered).numpy()
            assert sorted(allidx.tolist()) == list(range(len(lengths))), name
            for r in range(world):
                assert np.array_equal(gathered[r].numpy(), shards[r]), (name, r)
            cost = shard_cost(lengths, shards)
            biggest = int((lengths.astype(np.int64) ** 2).max())
            assert max(cost) - min(cost) <= biggest, (name, cost)
        results[rank] = True
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_partition_the_batch():
    world = 2
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    assert dict(results) == {0: True, 1: True}


def test_single_rank_and_edge_cases():
    assert [s.tolist() for s in shard_sequences([3, 1, 2], 1)] == [[0, 1, 2]]
    shards = shard_sequences([5, 5, 5, 5], 4)
    assert sorted(len(s) for s in shards) == [1, 1, 1, 1]
    shards = shard_sequences([], 3)
    assert all(s.size == 0 for s in shards)
    shards = shard_sequences([100, 1, 1, 1], 2)
    assert shard_cost([100, 1, 1, 1], shards) in ([10000, 3], [3, 10000])
