"""Data-parallel layout of the decode path over several GPUs.

Every head is independent in every call (a CTA or a warp works on one head at
a time, with no cross-head data), so the path shards by head with no collective
on the data path: each rank holds its own batch of requests, with the shapes of the
workload and its own seed, and runs the whole decode + recompression schedule
on them.  The only communication is for measurement: a barrier around the
timed region and the maximum of the ranks' times (weak scaling: the job's
throughput is all ranks' head-steps over the slowest rank's time).
"""
from __future__ import annotations

from typing import Optional

# Seeds of the ranks' batches: rank 0 keeps the workload's seed (so that one GPU
# runs exactly the named workload), rank k adds k times this odd stride.
SEED_STRIDE = 1_000_003


def shard(w, rank: int, world: int):
    """The workload of one rank: same shapes, an independent batch of requests."""
    if not 0 <= rank < world:
        raise ValueError(f'rank {rank} outside a world of {world}')
    return w if rank == 0 else w.with_(seed=w.seed + SEED_STRIDE * rank)


def job_heads(heads_per_rank: int, world: int) -> int:
    """Heads of the whole job (weak scaling: every rank holds the same count)."""
    return heads_per_rank * world


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over the ranks of the default process group (x itself
    without one).  ``device`` is where the reduction tensor lives: a CUDA device
    for NCCL, None (CPU) for gloo."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reports(rank: int) -> bool:
    """Whether this rank prints the job's result line (rank 0 only)."""
    return rank == 0


def barrier(device: Optional[int] = None) -> None:
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is None:
            dist.barrier()
        else:
            dist.barrier(device_ids=[device])
