"""Multi-process plumbing for running the op on several GPUs of one node.

The op has no exchange step: tokens are independent, so each rank owns its
own batch of tokens (its own seeded workload) and computes it alone; no
collective touches the data path.  The only collectives are the timing
barrier and the max-over-ranks of the measured time.
"""
from __future__ import annotations

import os


def env_world() -> tuple[int, int, int]:
    """(rank, local_rank, world_size) from the launcher's environment."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def init(backend: str) -> bool:
    """Initialise the default process group when launched with WORLD_SIZE > 1."""
    import torch.distributed as dist
    _, _, world = env_world()
    if world <= 1 or dist.is_initialized():
        return dist.is_initialized()
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return True


def shard_range(n: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous [start, end) of n units for this rank; sizes differ by at most one."""
    base, extra = divmod(n, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def rank_seed(seed: int, rank: int) -> int:
    """Seed of a rank's own batch (rank 0 keeps the workload's seed)."""
    return seed + 7919 * rank


def barrier(device=None) -> None:
    import torch.distributed as dist
    if dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not dist.is_initialized():
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not dist.is_initialized():
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())
