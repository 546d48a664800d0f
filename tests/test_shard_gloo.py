"""Multi-rank host logic on CPU (gloo, world size 2): the instance partition
covers every instance exactly once, and the timing reduction returns the
slowest rank's time on every rank."""

import os
import socket

import pytest
import torch.multiprocessing as mp

from kv_cache_eviction_snapkv_gb300 import shard


def test_shard_range_partition():
    for total in [0, 1, 7, 1024, 1025]:
        for world in [1, 2, 3, 8]:
            parts = shard.covers(total, world)
            flat = [i for p in parts for i in p]
            assert flat == list(range(total))
            sizes = [len(p) for p in parts]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard.shard_range(10, 2, 2)
    assert shard.rank_seed(1002, 0) == 1002 and shard.rank_seed(1002, 1) != 1002


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = shard.shard_range(1024, rank, world)
        t = shard.max_over_ranks(1.5 + rank)       # rank 1 is the slow one
        results[rank] = (mine.start, mine.stop, t)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_partition_and_max():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        got = dict(results)
    assert got[0][:2] == (0, 512) and got[1][:2] == (512, 1024)
    assert got[0][2] == got[1][2] == 2.5


def test_max_over_ranks_without_group():
    assert shard.max_over_ranks(3.25) == 3.25
