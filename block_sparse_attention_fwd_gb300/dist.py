"""Host-side helpers for running the path on several GPUs, one process each.

The BackLite path has no exchange step: the forward, the mask and the
backward of one (batch, kv-head group) touch only that group's Q/K/V/O/G_O
rows and produce only its outputs.  Ranks therefore split the groups among
themselves (no data-path collective) and only the timing is reduced (max over
ranks) for reporting.
"""
from __future__ import annotations


def shard_groups(B: int, Hk: int, rank: int, world: int):
    """The (batch, kv head) groups rank `rank` of `world` owns: round-robin over
    the B*Hk groups in (b, hk) order, so every group has exactly one owner."""
    if world < 1 or not (0 <= rank < world):
        raise ValueError("bad rank/world")
    return [divmod(u, Hk) for u in range(rank, B * Hk, world)]


def max_over_ranks(value: float, device=None) -> float:
    """Max of a float over all ranks of the default process group (identity
    when torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
