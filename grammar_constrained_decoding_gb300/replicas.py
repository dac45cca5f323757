"""Replica bookkeeping for running the decode step on several GPUs of one node.

Rows are independent, so the step shards by rows with no exchange: every GPU
holds its own grammar tables and mask cache and decodes its own B rows (weak
scaling).  The only cross-process traffic is outside the timed work: a barrier
on both sides of the timed region and a maximum over ranks of its duration.
"""

from __future__ import annotations

import os


def rank_info() -> tuple[int, int, int]:
    """(world size, rank, local rank) from the launcher's environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init(backend: str, device=None):
    """Joins the process group when launched with more than one rank; returns
    torch.distributed (or None for a single process)."""
    world, _, _ = rank_info()
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        if device is not None:
            dist.init_process_group(backend, device_id=device)
        else:
            dist.init_process_group(backend)
    return dist


def replica_seed(base: int, rank: int) -> int:
    """Seed of a replica's synthetic inputs: distinct per rank."""
    return base + 1000 * rank


def max_over_ranks(value: float, pg, device="cpu") -> float:
    """The largest value over all ranks (every rank gets it)."""
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, world: int, ms: float) -> float:
    """Units processed by all ranks per second, timed by the slowest rank."""
    return units_per_rank * world / (ms * 1e-3)
