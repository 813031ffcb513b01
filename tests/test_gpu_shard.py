"""A rank's share as strided views: the (batch, kv head) groups of
dist.shard_slices run as two "ranks" one after the other on one GPU, each
on slices of the full tensors (bl_shape strides, no gather), must give what
the unsharded call gives -- bit for bit for O, LSE, statistics, lists, G_K
and G_V, whose every value has one writer; G_Q within the reordering of its
fp32 reduce-adds.  Also a fused QKV projection (q, k, v as views of one
tensor) against the contiguous call.  Multi-GPU runs are not exercised here
(one GPU)."""
import pytest
import torch

from block_sparse_attention_fwd_gb300 import inputs
from block_sparse_attention_fwd_gb300.dist import shard_groups, shard_slices
from tests import parity_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__ as g
    g.build()


def _bits(t):
    t = t.detach()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    elif t.dtype == torch.float32:
        t = t.view(torch.int32)
    return t.cpu()


def _chain(shape, q, k, v, go, scale, negl, o, g_q, g_k, g_v):
    """forward (statistics) -> mask -> backward on the given (possibly strided)
    tensors; the per-call arrays (lse, statistics, lists) are its own."""
    from block_sparse_attention_fwd_gb300 import _lib
    dev = q.device
    T_r, T_c = _lib.tiles(shape)
    lse = torch.empty((shape.B, shape.H, shape.n), dtype=torch.float32, device=dev)
    stats = torch.empty((shape.B, shape.H, T_c, T_r * shape.block_q), dtype=torch.float32,
                        device=dev)
    _lib.attn_fwd(shape, q, k, v, scale, o, lse, stats)
    lists = _lib.alloc_lists(shape, dev)
    _lib.mask_from_stats(shape, stats, lse, negl, lists)
    ws = torch.empty(_lib.bwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)
    _lib.attn_bwd(shape, q, k, v, o, go, lse, scale, lists, g_q, g_k, g_v, ws)
    assert _lib.bwd_check_status(shape, ws) == 0
    return lse, stats, lists


CASES = [
    # kv heads split: each rank's q/k/v/o/gradients are head slices (strided)
    inputs.custom("shard_heads_n1000", B=2, n=1000, H=8, Hk=4, d=128, run=48, clusters=8,
                  alpha=3.0),
    # one kv head: batches split (contiguous slices)
    inputs.custom("shard_batches_n700", B=3, n=700, H=2, Hk=1, d=64, run=32, clusters=6,
                  alpha=3.0),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_two_ranks_of_slices_match_the_unsharded_call(w):
    from block_sparse_attention_fwd_gb300 import _lib
    negl = 0.05
    q, k, v, go = (x.cuda() for x in inputs.generate(w, seed=0))
    full = _lib.make_shape(w.B, w.n, w.H, w.Hk, w.d, w.block_q, w.block_k)
    o, gq, gk, gv = (torch.empty_like(x) for x in (q, q, k, v))
    lse, stats, lists = _chain(full, q, k, v, go, w.scale, negl, o, gq, gk, gv)

    G = w.H // w.Hk
    o2, gq2, gk2, gv2 = (torch.full_like(x, float("nan")) for x in (q, q, k, v))
    world = 2
    owned = []
    for rank in range(world):
        (b0, b1), (h0, h1) = shard_slices(w.B, w.Hk, rank, world)
        owned += shard_groups(w.B, w.Hk, rank, world)
        if b1 <= b0 or h1 <= h0:
            continue
        qs, os_, gos, gqs = (x[b0:b1, :, h0 * G:h1 * G] for x in (q, o2, go, gq2))
        ks, vs, gks, gvs = (x[b0:b1, :, h0:h1] for x in (k, v, gk2, gv2))
        shape = _lib.with_strides(
            _lib.make_shape(b1 - b0, w.n, (h1 - h0) * G, h1 - h0, w.d, w.block_q, w.block_k),
            q=qs, k=ks, v=vs, o=os_)
        lse_r, stats_r, lists_r = _chain(shape, qs, ks, vs, gos, w.scale, negl, os_, gqs, gks,
                                         gvs)
        hq = slice(h0 * G, h1 * G)
        assert torch.equal(_bits(lse_r), _bits(lse[b0:b1, hq]))
        assert torch.equal(_bits(stats_r), _bits(stats[b0:b1, hq]))
        for key in ("mask", "kv_idx", "kv_cnt", "q_idx", "q_cnt"):
            assert torch.equal(lists_r[key], lists[key][b0:b1, hq]), key
    assert sorted(owned) == [(b, h) for b in range(w.B) for h in range(w.Hk)]
    assert torch.equal(_bits(o2), _bits(o))
    assert torch.equal(_bits(gk2), _bits(gk)) and torch.equal(_bits(gv2), _bits(gv))
    assert U.rel_l2(U.cpu(gq2), U.cpu(gq)) <= 1e-3


def test_fused_qkv_views_match_contiguous_tensors():
    """q, k, v as head slices of one [B, n, H + 2 Hk, d] projection output, o
    and g_o as slices of wider buffers: the same results as contiguous copies."""
    from block_sparse_attention_fwd_gb300 import _lib
    w = inputs.custom("fused_qkv_n900", B=2, n=900, H=4, Hk=2, d=128, run=40, clusters=6,
                      alpha=3.0)
    q, k, v, go = (x.cuda() for x in inputs.generate(w, seed=4))
    qkv = torch.cat([q, k, v], dim=2)                 # [B, n, H + 2 Hk, d]
    qv, kv_, vv = qkv[:, :, :w.H], qkv[:, :, w.H:w.H + w.Hk], qkv[:, :, w.H + w.Hk:]
    wide_o = torch.empty((w.B, w.n, 2 * w.H, w.d), dtype=torch.bfloat16, device="cuda")
    wide_go = torch.zeros_like(wide_o)
    wide_go[:, :, w.H:] = go
    ov, gov = wide_o[:, :, :w.H], wide_go[:, :, w.H:]
    gqkv = torch.empty_like(qkv)
    gqv, gkv, gvv = gqkv[:, :, :w.H], gqkv[:, :, w.H:w.H + w.Hk], gqkv[:, :, w.H + w.Hk:]
    full = _lib.make_shape(w.B, w.n, w.H, w.Hk, w.d, 128, 128)
    shape = _lib.with_strides(full, q=qv, k=kv_, v=vv, o=ov)
    # q and g_q, k and g_k, v and g_v share strides here by construction
    assert gqv.stride() == qv.stride() and gkv.stride() == kv_.stride()
    assert gov.stride() == ov.stride()
    lse_s, stats_s, lists_s = _chain(shape, qv, kv_, vv, gov, w.scale, 0.05, ov, gqv, gkv, gvv)
    o, gq, gk, gv = (torch.empty_like(x) for x in (q, q, k, v))
    lse, stats, lists = _chain(full, q, k, v, go, w.scale, 0.05, o, gq, gk, gv)
    assert torch.equal(_bits(ov.contiguous()), _bits(o))
    assert torch.equal(_bits(lse_s), _bits(lse)) and torch.equal(_bits(stats_s), _bits(stats))
    assert torch.equal(lists_s["mask"], lists["mask"])
    assert torch.equal(_bits(gkv.contiguous()), _bits(gk))
    assert torch.equal(_bits(gvv.contiguous()), _bits(gv))
    assert U.rel_l2(U.cpu(gqv.contiguous()), U.cpu(gq)) <= 1e-3
