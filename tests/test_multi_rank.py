"""World-size-2 gloo run of the multi-rank host logic (CPU only): the group
partition covers every (batch, kv head) group exactly once with no data-path
collective, and the timing reduction takes the max over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from block_sparse_attention_fwd_gb300.dist import max_over_ranks, shard_groups


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
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        t = max_over_ranks(10.0 + rank)
        out[rank] = (gathered, t)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("B,Hk", [(1, 40), (2, 8), (3, 1)])
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


def test_single_process_identity():
    assert shard_groups(2, 3, 0, 1) == [(0, 0), (0, 1), (0, 2), (1, 0), (1, 1), (1, 2)]
    assert max_over_ranks(3.5) == 3.5
    with pytest.raises(ValueError):
        shard_groups(1, 1, 2, 2)
