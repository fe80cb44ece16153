"""Multi-process helpers for replica runs (one process per GPU).

The layer runs as independent replicas: each rank processes its own units and
no collective sits on the data path.  The only cross-rank steps are a barrier
around the timed region and the reduction of the per-rank step time to the
slowest rank, which both work on any torch.distributed backend (NCCL on GPUs,
gloo on CPU for the tests).
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def max_over_ranks(value: float, device: torch.device | str = "cpu") -> float:
    """The largest `value` over all ranks (the value itself without a process group)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, ms_per_step_max: float, world: int) -> float:
    """Whole-job throughput: the units all ranks processed in one step divided by
    the slowest rank's step time (units per second)."""
    if ms_per_step_max <= 0:
        raise ValueError("step time must be positive")
    return world * units_per_rank / (ms_per_step_max * 1e-3)
