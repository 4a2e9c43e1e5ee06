"""Replica bookkeeping for multi-GPU runs of the decode benchmark.

The decode work shards by (sequence, KV head) with no exchange between GPUs, so N GPUs
run N independent replicas: each rank times its own steps, the job's step time is the
maximum over ranks, and the job's throughput is all ranks' bytes over that time.
"""
from __future__ import annotations

import torch


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of `value` over the ranks of the default process group (itself if none)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank: float, ms_per_step_max: float, world_size: int) -> float:
    """Whole-job GB/s: every rank moves `bytes_per_rank` per step; the slowest rank sets the time."""
    return bytes_per_rank * world_size / (ms_per_step_max * 1e-3) / 1e9
