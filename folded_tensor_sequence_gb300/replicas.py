"""Multi-process bookkeeping of the throughput run: one process per GPU, each a
full replica of the layer on its own batch (the layer's work units -- whole
sequences -- are independent, so nothing on the data path is exchanged).

Ranks meet only around the timed region: a barrier before and after it, and a
max-reduction of the elapsed times, so the whole job is as slow as its slowest
rank.  Works with any torch.distributed backend (nccl on GPUs, gloo on CPU).
"""

from __future__ import annotations

import os
from dataclasses import dataclass


@dataclass(frozen=True)
class RankEnv:
    world_size: int
    rank: int
    local_rank: int


def rank_env(env=None) -> RankEnv:
    """World size, rank and local rank as torchrun exports them (1, 0, 0 alone)."""
    env = os.environ if env is None else env
    return RankEnv(int(env.get("WORLD_SIZE", "1")), int(env.get("RANK", "0")), int(env.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks (the local value when not distributed)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world_size: int, units_per_step: float, steps: int, elapsed_ms: float) -> float:
    """Units per second of the whole job: every rank processed `units_per_step`
    per step, and the job took the slowest rank's `elapsed_ms`."""
    if elapsed_ms <= 0:
        raise ValueError("elapsed time must be positive")
    return world_size * units_per_step * steps / (elapsed_ms / 1e3)
