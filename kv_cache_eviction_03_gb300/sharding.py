"""Splitting independent (batch, head) pairs across ranks.

Pairs never interact in H2O (eviction is decided per head, batch rows are
independent), so ranks need no exchange on the data path: each one runs a
contiguous range of heads (or batch rows) in its own cache, and the only
collective is the scalar max used to time the slowest rank.
"""
from __future__ import annotations


def shard_range(n: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous [lo, hi) share of n items for `rank` (sizes differ by <= 1)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    base, extra = divmod(n, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def max_over_ranks(values, dist=None, device=None):
    """Element-wise max of a list of floats over all ranks (identity when
    torch.distributed is not initialised)."""
    if dist is None or not dist.is_available() or not dist.is_initialized():
        return list(values)
    import torch

    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()
