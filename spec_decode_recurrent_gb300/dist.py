"""Process-group plumbing for running one independent replica per GPU.

The path has no exchange step: value heads, rows and layers are independent
and every rank already holds its accepted lengths after sampling, so N GPUs
run N independent steps (weak scaling).  The only cross-rank traffic is the
benchmark's barrier and the max-over-ranks reduction of its timings.
"""
from __future__ import annotations

import os
from typing import Tuple

import torch
import torch.distributed as dist


def world() -> Tuple[int, int, int]:
    """(rank, local_rank, world_size) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def init(backend: str = "nccl") -> Tuple[int, int, int]:
    rank, local_rank, world_size = world()
    if world_size > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world_size)
    return rank, local_rank, world_size


def replica_seed(base: int, rank: int) -> int:
    """Each replica draws its own inputs of the same shape."""
    return int(base) + 1000 * int(rank)


def barrier() -> None:
    if dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    if not (dist.is_initialized() and dist.get_world_size() > 1):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def finalize() -> None:
    if dist.is_initialized():
        dist.destroy_process_group()
