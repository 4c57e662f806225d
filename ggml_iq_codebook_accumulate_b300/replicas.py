"""Replica runs on several GPUs of one node.

Blocks, vectors and the imatrix pass of one weight are independent of every other weight's, so a
job over N GPUs runs N replicas of the hot path, one process per GPU, each on its own batch.  No
data crosses ranks: the only traffic is host-side bookkeeping, a barrier around the timed region
and the maximum of the ranks' step times (the job is as fast as its slowest rank).  The job's
throughput counts the units every rank processed (weak scaling: the work per GPU is fixed).
"""
from __future__ import annotations

import os


def world_info():
    """(rank, world_size, local_rank) from the launcher's environment; (0, 1, 0) when run alone."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def _initialized():
    import torch.distributed as dist
    return dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1


def barrier():
    """Barrier over all ranks (no-op when run alone)."""
    if _initialized():
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, device=None) -> float:
    """The largest of the ranks' values, on every rank.  `device` is where the reduction tensor
    lives: a CUDA device for NCCL, None (CPU) for gloo."""
    if not _initialized():
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, seconds: float, world: int) -> float:
    """Units per second of the whole job: every rank's units over the slowest rank's time."""
    if seconds <= 0 or world < 1:
        raise ValueError("seconds must be positive and world at least 1")
    return world * units_per_rank / seconds
