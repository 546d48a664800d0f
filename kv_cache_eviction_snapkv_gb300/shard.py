"""Multi-GPU host logic: every (layer, sequence, head) instance is independent
(the SnapKV page selects per layer and per head), so ranks share no data and
exchange nothing on the data path. Weak scaling: rank r processes its own
batch of instances (shard r of an N-times larger batch); the only collective
is the benchmark's max over the ranks' timings.
"""

from __future__ import annotations

from typing import List


def shard_range(total: int, rank: int, world: int) -> range:
    """Contiguous, balanced partition of `total` instances: sizes differ by <= 1."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    base, extra = divmod(total, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))


def rank_seed(seed: int, rank: int) -> int:
    """Input seed of rank r's batch (rank 0 keeps the workload's own seed)."""
    return seed + 7919 * rank


def max_over_ranks(value: float, device=None) -> float:
    """The largest value over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def covers(total: int, world: int) -> List[range]:
    return [shard_range(total, r, world) for r in range(world)]
