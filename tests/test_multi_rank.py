"""World-size-2 gloo run of the multi-rank host logic (CPU only): the group
partition covers every (batch, kv head) group exactly once with no data-path
collective, and the timing reduction takes the max over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from block_sparse_attention_fwd_gb300.dist import max_over_ranks, shard_groups, shard_slices


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, B, Hk, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        mine = shard_groups(B, Hk, rank, world)
        (b0, b1), (h0, h1) = shard_slices(B, Hk, rank, world)
        # the rank's slices hold exactly its groups
        assert mine == [(b, h) for b in range(b0, b1) for h in range(h0, h1)]
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        t = max_over_ranks(10.0 + rank)
        out[rank] = (gathered, t)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("B,Hk", [(1, 40), (2, 8), (3, 1), (2, 5), (1, 1)])
def test_two_gloo_ranks_partition_and_time(B, Hk):
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), B, Hk, out), nprocs=world,
                       join=True, start_method="spawn")
    for rank in range(world):
        gathered, t = out[rank]
        allg = [g for part in gathered for g in part]
        assert sorted(allg) == [(b, h) for b in range(B) for h in range(Hk)]
        assert len(allg) == len(set(allg))
        assert t == 11.0


def test_shard_slices_are_balanced_blocks():
    # kv heads split when there are enough, batches otherwise
    assert [shard_slices(1, 40, r, 2) for r in range(2)] == [((0, 1), (0, 20)), ((0, 1), (20, 40))]
    assert [shard_slices(2, 5, r, 2) for r in range(2)] == [((0, 2), (0, 3)), ((0, 2), (3, 5))]
    assert [shard_slices(3, 1, r, 2) for r in range(2)] == [((0, 2), (0, 1)), ((2, 3), (0, 1))]
    assert [shard_slices(1, 8, r, 3) for r in range(3)] == [((0, 1), (0, 3)), ((0, 1), (3, 6)),
                                                           ((0, 1), (6, 8))]
    assert shard_groups(1, 1, 1, 2) == []          # more ranks than groups: rank 1 idle


def test_single_process_identity():
    assert shard_groups(2, 3, 0, 1) == [(0, 0), (0, 1), (0, 2), (1, 0), (1, 1), (1, 2)]
    assert max_over_ranks(3.5) == 3.5
    with pytest.raises(ValueError):
        shard_groups(1, 1, 2, 2)


def _seq_worker(rank, world, port, cu, causal, out):
    from block_sparse_attention_fwd_gb300.dist import shard_sequences
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        mine, local, ranges = shard_sequences(cu, rank, world, causal=causal)
        gathered = [None] * world
        dist.all_gather_object(gathered, (mine, local, ranges))
        out[rank] = gathered
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("causal", [False, True])
def test_two_gloo_ranks_shard_packed_sequences(causal):
    """Every sequence of a packed batch has exactly one owner, all ranks agree
    on the assignment, each rank's local packing holds its sequences' tokens,
    and the work is balanced to within the largest sequence."""
    from block_sparse_attention_fwd_gb300.dist import sequence_work
    from block_sparse_attention_fwd_gb300.inputs import document_lengths
    lengths = document_lengths(65536, seed=3)
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_seq_worker, args=(world, _free_port(), cu, causal, out), nprocs=world,
                       join=True, start_method="spawn")
    assert out[0] == out[1]                         # the same assignment on every rank
    parts = out[0]
    owned = [s for mine, _, _ in parts for s in mine]
    assert sorted(owned) == list(range(len(lengths)))
    loads = []
    for mine, local, ranges in parts:
        assert local[-1] == sum(b - a for a, b in ranges)
        assert [b - a for a, b in ranges] == [lengths[s] for s in mine]
        loads.append(sum(sequence_work(lengths[s], causal) for s in mine))
    assert max(loads) - min(loads) <= max(sequence_work(n, causal) for n in lengths)


def test_sequence_shards_single_process():
    from block_sparse_attention_fwd_gb300.dist import sequence_work, shard_sequences
    assert shard_sequences([0, 5, 5, 9], 0, 1) == ([0, 1, 2], [0, 5, 5, 9],
                                                  [(0, 5), (5, 5), (5, 9)])
    assert sequence_work(4) == 16 and sequence_work(4, causal=True) == 10
    assert sequence_work(10, causal=True, window=3) == 6 + 7 * 3
    with pytest.raises(ValueError):
        shard_sequences([1, 5], 0, 1)
    with pytest.raises(ValueError):
        shard_sequences([0, 5], 1, 1)
