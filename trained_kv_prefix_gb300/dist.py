"""Data-parallel plumbing for cartridge training and serving (host side).

One process per GPU.  Training shards the packed batch of sequences across
ranks; every rank holds a replica of the cartridge, so the only exchange is
the sum of the cartridge gradients (the batch sum that one GPU does inside
its dK/dV kernel becomes a cross-rank all-reduce).  Serving shards the
conversations across ranks with the cartridge replicated: no exchange.
"""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def env_rank_world():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_from_env(backend: str) -> bool:
    """Initialise the default process group when launched with WORLD_SIZE > 1.
    Returns True when a group exists."""
    _, world, _ = env_rank_world()
    if world <= 1:
        return False
    if not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return True


def shard(total: int, rank: int, world: int):
    """Contiguous [lo, hi) slice of `total` items owned by `rank`."""
    base, extra = divmod(total, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def allreduce_cartridge_grads(dkc: torch.Tensor, dvc: torch.Tensor) -> None:
    """Sum the per-rank cartridge gradients in place (frozen rows stay 0
    because every rank writes exact zeros there)."""
    if dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(dkc, op=dist.ReduceOp.SUM)
        dist.all_reduce(dvc, op=dist.ReduceOp.SUM)


def max_over_ranks(values, device) -> list:
    """Element-wise maximum of a list of floats over all ranks."""
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def barrier(device=None) -> None:
    if dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and torch.device(device).type == "cuda":
            dist.barrier(device_ids=[torch.device(device).index])
        else:
            dist.barrier()
