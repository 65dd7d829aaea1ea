"""Host logic for running the verify decode on several GPUs (one process per
GPU).  The sequences of a batch are independent, so a global batch is split
into contiguous sequence ranges, one per rank, with no exchange on the data
path; the only collective is the max-over-ranks of the measured time."""

from __future__ import annotations

from typing import Tuple


def shard(n_total: int, rank: int, world: int) -> Tuple[int, int]:
    """Contiguous [start, end) sequence range of `rank`; the first
    n_total % world ranks take one extra sequence."""
    if world < 1 or not 0 <= rank < world or n_total < 0:
        raise ValueError("bad shard arguments")
    base, extra = divmod(n_total, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of `value` over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
