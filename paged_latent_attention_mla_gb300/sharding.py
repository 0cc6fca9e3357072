"""Multi-GPU layout: requests are independent, so N GPUs take N disjoint shards.

Decode rows of different requests never interact, so the batch partitions by
request with no data-path collective: rank k of N decodes requests
[start_k, end_k).  Timing across ranks takes the maximum (the slowest rank ends
the step); that reduction is the only collective and it sits outside the path.
"""

from __future__ import annotations

import torch


def shard_rows(B: int, world: int, rank: int) -> tuple:
    """Contiguous, balanced request range [start, end) of `rank` among `world` ranks."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world / rank")
    base, extra = divmod(B, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def rank_seed(seed: int, rank: int) -> int:
    """Seed of rank's own batch when every rank decodes a full batch (weak scaling)."""
    return seed + 1000003 * rank


def max_over_ranks(value: float) -> float:
    """Maximum of a host scalar over all ranks (identity when not distributed)."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
