"""Multi-GPU bookkeeping of the benchmark: one process per GPU, each with its own
independent decode workload (sequences never span GPUs, so there is no data
exchange), timed together with the slowest rank deciding the step time."""

from __future__ import annotations

import os

import torch
import torch.distributed as dist

# Seeds of different ranks' instances are spaced by a prime so no two ranks draw
# the same inputs.
RANK_SEED_STRIDE = 7919


def world() -> tuple[int, int, int]:
    """(rank, world size, local rank) from the torchrun environment (1 GPU: 0, 1, 0)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(base_seed: int, rank: int) -> int:
    return base_seed + RANK_SEED_STRIDE * rank


def max_over_ranks(value: float, device: torch.device) -> float:
    """The largest value over all ranks (the identity without a process group)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_rate(bytes_per_rank: int, world_size: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's step time."""
    return world_size * bytes_per_rank / (ms_per_step * 1e-3) / 1e9
