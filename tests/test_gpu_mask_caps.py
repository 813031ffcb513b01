"""The mask pass at every key-tile capacity of its kernel (256, 512, 1024 and
2048 key tiles per row).  The selection depends only on the statistics and
the LSE it is given, so the inputs are synthetic statistics drawn on the
GPU: each row puts its weight on a few key tiles near a row-dependent
centre.  Sampled query tiles are compared bit for bit with the oracle's rule
applied to the same values; the transposed lists are checked against the
whole GPU mask."""
import numpy as np
import pytest
import torch

from oracle import mask_spec as M
from tests import parity_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__ as g
    g.build()


CASES = [
    # (n, block_q, block_k) -> T_c
    (5000, 64, 64),        # 79   -> capacity 256
    (40000, 128, 128),     # 313  -> 512
    (40000, 128, 64),      # 625  -> 1024
    (131000, 128, 64),     # 2047 -> 2048
]


def _stats(n, H, bq, bk, seed):
    """stats [1,H,T_c,T_r*bq] fp32 and lse [1,H,n]: row r favours key tiles
    near a centre that moves with r, plus noise; rows >= n are -inf."""
    T_r, T_c = -(-n // bq), -(-n // bk)
    g = torch.Generator(device="cuda").manual_seed(seed)
    r = torch.arange(T_r * bq, device="cuda", dtype=torch.float32)
    j = torch.arange(T_c, device="cuda", dtype=torch.float32)
    stats = torch.empty((1, H, T_c, T_r * bq), dtype=torch.float32, device="cuda")
    for h in range(H):
        centre = (r * (T_c / (T_r * bq)) * (1 + 0.3 * h)) % T_c
        dist = (j[:, None] - centre[None, :]).abs()
        s = -0.8 * dist + 2.0 * torch.randn((T_c, T_r * bq), generator=g, device="cuda")
        s[:, n:] = -float("inf")
        stats[0, h] = s
        del dist, s
    lse = torch.logsumexp(stats[:, :, :, :n], dim=2).contiguous()      # [1,H,n]
    return stats, lse


@pytest.mark.parametrize("n,bq,bk", CASES)
def test_mask_capacity_paths_match_oracle(n, bq, bk):
    from block_sparse_attention_fwd_gb300 import _lib
    H, negl = 2, 0.05
    shape = _lib.make_shape(1, n, H, H, 64, bq, bk)
    T_r, T_c = _lib.tiles(shape)
    stats, lse = _stats(n, H, bq, bk, seed=n + bk)
    lists = U.gpu_mask(shape, stats, lse, negl)
    mask = U.cpu(lists["mask"])
    kv_idx, kv_cnt = U.cpu(lists["kv_idx"]), U.cpu(lists["kv_cnt"])
    rng = np.random.default_rng(bk)
    tiles = sorted(set([0, T_r - 1] + rng.integers(0, T_r, size=10).tolist()))
    T = M.threshold(negl)
    for h in range(H):
        for i in tiles:
            rows = slice(i * bq, (i + 1) * bq)
            st = U.cpu(stats[0, h, :, rows])                       # [T_c, bq]
            nrow = min(n - i * bq, bq)
            lr = np.zeros(bq, dtype=np.float32)
            lr[:nrow] = U.cpu(lse[0, h, i * bq:i * bq + nrow])
            d = M.tile_weights(st, lr, nrow, bq)                    # [1, T_c]
            want, _ = M.select_row(d[0], T)
            assert np.array_equal(mask[0, h, i], want), (h, i)
            kept = np.nonzero(want)[0]
            assert kv_cnt[0, h, i] == len(kept)
            assert np.array_equal(kv_idx[0, h, i, :len(kept)], kept)
    assert 0 < mask.sum() < mask.size
    ref = M.lists_from_mask(mask)
    assert np.array_equal(U.cpu(lists["q_cnt"]), ref["q_cnt"])
    q_idx, q_cnt = U.cpu(lists["q_idx"]), ref["q_cnt"]
    for h in range(H):
        for jj in range(0, T_c, max(1, T_c // 64)):
            c = q_cnt[0, h, jj]
            assert np.array_equal(q_idx[0, h, jj, :c], ref["q_idx"][0, h, jj, :c]), (h, jj)
