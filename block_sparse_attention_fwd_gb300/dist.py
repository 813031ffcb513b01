"""Host-side helpers for running the path on several GPUs, one process each.

The BackLite path has no exchange step: the forward, the mask and the
backward of one (batch, kv-head group) touch only that group's Q/K/V/O/G_O
rows and produce only its outputs.  Ranks therefore split the groups among
themselves (no data-path collective) and only the timing is reduced (max over
ranks) for reporting.
"""
from __future__ import annotations


def _block(count: int, rank: int, world: int):
    """[lo, hi) of rank's balanced contiguous block of `count` items."""
    base, extra = divmod(count, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def shard_slices(B: int, Hk: int, rank: int, world: int):
    """The rectangle of (batch, kv head) groups rank `rank` of `world` owns:
    ((b0, b1), (hk0, hk1)).  Kv heads are split into balanced contiguous blocks
    when there are at least as many as ranks, batches otherwise, so a rank's
    share of every tensor is one slice -- q[b0:b1, :, hk0*G:hk1*G] and
    k[b0:b1, :, hk0:hk1] with G = H / Hk -- that the library takes as a strided
    view (bl_shape strides), with no gather.  Every group has exactly one
    owner; a rank may own none when there are more ranks than groups."""
    if world < 1 or not (0 <= rank < world):
        raise ValueError("bad rank/world")
    if Hk >= world:
        return (0, B), _block(Hk, rank, world)
    return _block(B, rank, world), (0, Hk)


def shard_groups(B: int, Hk: int, rank: int, world: int):
    """The (batch, kv head) groups of shard_slices, in (b, hk) order."""
    (b0, b1), (h0, h1) = shard_slices(B, Hk, rank, world)
    return [(b, hk) for b in range(b0, b1) for hk in range(h0, h1)]


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


def sequence_work(n: int, causal: bool = False, window: int = 0) -> int:
    """(query, key) pairs of one sequence of length n that attend: the work of
    its forward and backward up to a constant."""
    if not causal:
        return n * n
    if not window or window >= n:
        return n * (n + 1) // 2
    return window * (window + 1) // 2 + (n - window) * window


def shard_sequences(cu_seqlens, rank: int, world: int, causal: bool = False, window: int = 0):
    """The sequences of a packed batch that rank `rank` of `world` owns.

    Sequences carry no exchange either: each attends only to itself.  They go,
    largest work first (ties by index), to the rank with the least work so far
    (ties to the lower rank), so every rank derives the same assignment from
    cu_seqlens alone and each sequence has exactly one owner.  Returns
    (seq_ids ascending, local cu_seqlens of the owned sequences packed in that
    order, their token ranges [(start, end)] in the global packing)."""
    if world < 1 or not (0 <= rank < world):
        raise ValueError("bad rank/world")
    cu = [int(x) for x in cu_seqlens]
    if not cu or cu[0] != 0 or any(b < a for a, b in zip(cu[:-1], cu[1:])):
        raise ValueError("cu_seqlens must start at 0 and be non-decreasing")
    lengths = [b - a for a, b in zip(cu[:-1], cu[1:])]
    order = sorted(range(len(lengths)),
                   key=lambda s: (-sequence_work(lengths[s], causal, window), s))
    load = [0] * world
    owner = [0] * len(lengths)
    for s in order:
        r = min(range(world), key=lambda x: (load[x], x))
        owner[s] = r
        load[r] += sequence_work(lengths[s], causal, window)
    mine = [s for s in range(len(lengths)) if owner[s] == rank]
    local = [0]
    for s in mine:
        local.append(local[-1] + lengths[s])
    return mine, local, [(cu[s], cu[s + 1]) for s in mine]
