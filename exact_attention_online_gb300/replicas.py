"""Host-side logic of the multi-GPU (replica) benchmark.

The attention path shards with no data-path exchange: batches, and the
(batch, kv-head) groups inside a batch, are independent in the forward and
the backward, and the GQA sums of dK/dV stay inside a group.  N GPUs therefore
run N independent problems of the same per-GPU size (weak scaling); the only
collectives are the benchmark's barrier and its max-over-ranks of the timed
interval.  These helpers hold that logic so it can be tested with the gloo
backend on CPU.
"""
from __future__ import annotations

import os

# Seed stride between ranks: each rank draws its own batch.
RANK_SEED_STRIDE = 7919


def dist_env() -> tuple[int, int, int]:
    """(world_size, rank, local_rank) from the torchrun environment."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_workload(w, rank: int):
    """The workload rank `rank` runs: same shapes, its own seed."""
    return w.with_(seed=w.seed + RANK_SEED_STRIDE * rank)


def max_over_ranks(value: float, device=None) -> float:
    """Max of `value` over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(work_per_step: float, steps: int, world_size: int, ms_total: float) -> float:
    """Units per second of the whole job: every rank did `steps` steps of
    `work_per_step` units; the job took the slowest rank's `ms_total`."""
    if ms_total <= 0:
        raise ValueError("elapsed time must be positive")
    return work_per_step * steps * world_size / (ms_total * 1e-3)
