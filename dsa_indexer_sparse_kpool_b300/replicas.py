"""Running the DSA step on several GPUs as independent replicas.

The step is data-parallel over sequences: each rank runs its own batch, drawn
with its own seed, and nothing crosses between ranks on the data path.  The
only communication is host-side bookkeeping of the measurement: a barrier
around the timed region and the maximum of the ranks' times, so the whole
job's throughput is (units on all ranks) / (slowest rank's time).
"""
from __future__ import annotations

from typing import List, Sequence

import torch
import torch.distributed as dist

RANK_SEED_STRIDE = 1000


def rank_seed(base_seed: int, rank: int) -> int:
    """Seed of `rank`'s batch: distinct per rank, the same on every run."""
    return int(base_seed) + RANK_SEED_STRIDE * int(rank)


def distributed() -> bool:
    return dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1


def barrier() -> None:
    if distributed():
        dist.barrier()


def max_over_ranks(values: Sequence[float], device=None) -> List[float]:
    """Element-wise maximum of `values` over all ranks (identity on one rank)."""
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if distributed():
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_rate(units_per_rank: int, world: int, seconds: float) -> float:
    """Whole-job throughput when every rank processed `units_per_rank` units and
    the slowest rank took `seconds`."""
    return float(units_per_rank) * int(world) / float(seconds)
