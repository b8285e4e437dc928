"""Host-side helpers for running the operator on several GPUs.

The operator is independent per (batch, head) pair, so a job partitions over
B x H with no exchange inside the operator; the only cross-rank step is the
benchmark's max-over-ranks of a timing.
"""
from __future__ import annotations

from typing import List, Tuple


def head_partition(B: int, H: int, world: int, rank: int) -> Tuple[int, int]:
    """Contiguous [start, end) range of flattened (b, h) heads owned by `rank`.

    Every head belongs to exactly one rank; sizes differ by at most one."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError(f"bad rank {rank} of {world}")
    n = B * H
    base, extra = divmod(n, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def heads_of(B: int, H: int, world: int, rank: int) -> List[Tuple[int, int]]:
    s, e = head_partition(B, H, world, rank)
    return [(i // H, i % H) for i in range(s, e)]


def max_over_ranks(values, device=None):
    """Elementwise max of a list of floats over all ranks (identity without a
    process group)."""
    import torch
    import torch.distributed as dist

    vals = [float(v) for v in values]
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return vals
    t = torch.tensor(vals, dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]
