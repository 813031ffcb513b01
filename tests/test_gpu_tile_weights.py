"""Tile weights reduced in the forward (bl_attn_fwd_tile_weights) and the
mask built from them (bl_mask_from_tile_weights), against the oracle's
reduction of the GPU's own statistics ("BackLite" README, How It Works,
Phase 2: p_tile = exp(LSE_tile - LSE_row)), bit for bit.

Every case runs the forward three ways -- plain, with statistics and tile
weights, and with tile weights only (statistics rows in the scratch slots)
-- and checks that O, LSE and the statistics do not change, that the tile
weights equal the oracle's d_ij of the returned statistics exactly and do
not depend on whether statistics are returned, and that the lists built
from the weights equal the lists bl_mask_from_stats builds, and the
oracle's."""
import numpy as np
import pytest
import torch

from block_sparse_attention_fwd_gb300 import inputs
from oracle import mask_spec as M
from tests import parity_util as U

pytestmark = pytest.mark.gpu

CASES = [
    inputs.custom("tw_ragged_n1000_d128_gqa", B=2, n=1000, H=4, Hk=2, d=128, run=48,
                  clusters=8, alpha=3.0),
    inputs.custom("tw_ragged_n300_d128", B=1, n=300, H=3, Hk=1, d=128, run=16, clusters=4,
                  alpha=2.0),
    inputs.WORKLOADS["clustered_n4096_d64"],
    inputs.custom("tw_causal_n1500_d128", B=1, n=1500, H=4, Hk=2, d=128, run=32, clusters=8,
                  alpha=3.0, causal=True),
    # 64-wide tiles: odd T_r (the last 128-row MMA tile reaches past the
    # statistics' rows), both mixed shapes
    inputs.custom("tw_q64k64_n777_d64", B=1, n=777, H=2, Hk=1, d=64, block_q=64, block_k=64,
                  run=32, clusters=6, alpha=2.5),
    inputs.custom("tw_q64k128_n130_d128", B=2, n=130, H=2, Hk=2, d=128, block_q=64,
                  block_k=128, run=16, clusters=3, alpha=2.0),
    inputs.custom("tw_q128k64_n700_d64_gqa", B=1, n=700, H=4, Hk=2, d=64, block_q=128,
                  block_k=64, run=40, clusters=5, alpha=3.0),
    inputs.custom("tw_window_n2000_d64", B=1, n=2000, H=2, Hk=1, d=64, run=32, clusters=8,
                  alpha=3.0, causal=True, window=300),
]


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__ as g
    g.build()


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int32).numpy()


def _same_bits(a, b):
    return np.array_equal(_bits(a), _bits(b))


def _oracle_logw(stats, lse, w):
    st, ls = U.cpu(stats), U.cpu(lse)
    return np.stack([np.stack([M.tile_weights(st[b, h], ls[b, h], w.n, w.block_q)
                               for h in range(w.H)]) for b in range(w.B)])


def run_three_ways(w, shape, q, k, v):
    from block_sparse_attention_fwd_gb300 import _lib
    qd, kd, vd, o, lse, stats = U.gpu_forward(shape, q, k, v, w.scale)
    T_r, T_c = _lib.tiles(shape)
    o1, lse1 = torch.empty_like(o), torch.empty_like(lse)
    st1 = torch.empty_like(stats)
    lw1 = torch.empty((w.B, w.H, T_r, T_c), dtype=torch.float32, device=o.device)
    _lib.attn_fwd_tile_weights(shape, qd, kd, vd, w.scale, o1, lse1, lw1, tile_stats=st1)
    o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
    lw2 = torch.full_like(lw1, float("nan"))
    ws = torch.empty(_lib.fwd_workspace_bytes(shape), dtype=torch.uint8, device=o.device)
    _lib.attn_fwd_tile_weights(shape, qd, kd, vd, w.scale, o2, lse2, lw2, workspace=ws)
    torch.cuda.synchronize()
    return (o, lse, stats), (o1, lse1, st1, lw1), (o2, lse2, lw2)


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_tile_weights_match_the_oracle_and_the_stats_path(w):
    from block_sparse_attention_fwd_gb300 import _lib
    q, k, v, _ = inputs.generate(w, seed=0)
    shape = _lib.make_shape(w.B, w.n, w.H, w.Hk, w.d, w.block_q, w.block_k, w.causal, w.window)
    (o, lse, stats), (o1, lse1, st1, lw1), (o2, lse2, lw2) = run_three_ways(w, shape, q, k, v)
    # the reduction changes nothing else the forward writes
    assert _same_bits(o, o1) and _same_bits(o, o2)
    assert _same_bits(lse, lse1) and _same_bits(lse, lse2)
    assert _same_bits(stats, st1)
    # d_ij: the oracle's reduction of the GPU's own statistics, bit for bit;
    # and the same whether or not the statistics are returned
    ref = _oracle_logw(st1, lse1, w)
    assert np.array_equal(U.cpu(lw1), ref, equal_nan=True)
    assert _same_bits(lw1, lw2)
    for negl in (0.0, 0.05, 0.3):
        a = _lib.alloc_lists(shape, o.device)
        _lib.mask_from_tile_weights(shape, lw2, negl, a)
        b = U.gpu_mask(shape, stats, lse, negl)
        for key in ("mask", "kv_idx", "kv_cnt", "q_idx", "q_cnt"):
            assert torch.equal(a[key], b[key]), (key, negl)
        assert int(a["nan_count"].item()) == int(b["nan_count"].item())
        ref_lists = M.mask_from_stats(U.cpu(st1), U.cpu(lse1), w.n, w.block_q, w.block_k, negl,
                                      w.causal, w.window)
        U.assert_lists_equal(a, ref_lists)


@pytest.mark.parametrize("n", [1024, 640, 32768, 38400, 128000, 262144])
def test_tile_weights_mask_on_planted_weights(n):
    """Hand-built weights with ties, -inf and NaN tiles: the mask from the
    weights is the oracle's selection of exactly those rows.  T_c = 5, 8,
    256, 300, 1000 and 2048 run the one-warp-per-row kernel with 8, 16, 32
    and 64 entries per lane."""
    from block_sparse_attention_fwd_gb300 import _lib
    B, H = 1, 2
    shape = _lib.make_shape(B, n, H, H, 128, 128, 128)
    T = n // 128
    rng = np.random.default_rng(11)
    d = np.log(rng.dirichlet(np.full(T, 0.4), size=(B, H, T))).astype(np.float32)
    d = np.minimum(d, 0).astype(np.float32)
    d[0, 0, 2, 1] = d[0, 0, 2, 0]                 # tie
    d[0, 1, 3, min(5, T - 1)] = -np.inf          # empty tile
    d[0, 1, 4, min(6, T - 2)] = np.nan           # NaN weight
    lw = torch.from_numpy(d).cuda()
    for negl in (0.0, 0.02, 0.2, 0.9):
        lists = _lib.alloc_lists(shape, "cuda")
        _lib.mask_from_tile_weights(shape, lw, negl, lists)
        Tn = M.threshold(negl)
        mask = np.zeros((B, H, T, T), dtype=np.uint8)
        nans = 0
        for h in range(H):
            for i in range(T):
                mask[0, h, i], c = M.select_row(d[0, h, i], Tn)
                nans += c
        U.assert_lists_equal(lists, M.lists_from_mask(mask))
        assert int(lists["nan_count"].item()) == nans


def test_tile_weights_rejects_what_it_does_not_build():
    from block_sparse_attention_fwd_gb300 import _lib
    wide = _lib.make_shape(1, 2049 * 64, 1, 1, 64, 64, 64)     # T_c = 2049
    assert _lib.fwd_workspace_bytes(wide) == 0
    big = _lib.make_shape(1, 2049 * 128, 1, 1, 128, 128, 128)    # T_c > 2048
    assert _lib.fwd_workspace_bytes(big) == 0
    s = _lib.make_shape(1, 512, 2, 1, 128, 128, 128)
    assert _lib.fwd_workspace_bytes(s) > 0
