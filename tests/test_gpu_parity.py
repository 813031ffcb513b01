"""GPU parity of the whole hot path against the fp64 oracle, element by
element, on cases the oracle finishes in seconds (several tiles, ragged
tails, GQA, both head dims, both tile sizes).  Every call goes through the
C ABI binding."""
import numpy as np
import pytest
import torch

from block_sparse_attention_fwd_gb300 import inputs
from oracle import attention as A
from tests import parity_util as U

pytestmark = pytest.mark.gpu

CASES = [
    (inputs.WORKLOADS["tiny_n256_d64"], 0.0),
    (inputs.WORKLOADS["tiny_n256_d64"], 0.05),
    (inputs.custom("ragged_n1000_d128_gqa", B=2, n=1000, H=4, Hk=2, d=128, run=48,
                   clusters=8, alpha=3.0), 0.05),
    (inputs.custom("ragged_n777_d64_t64", B=1, n=777, H=2, Hk=1, d=64, block_q=64,
                   block_k=64, run=32, clusters=6, alpha=2.5), 0.1),
    (inputs.custom("mixed_n640_d128_q64k128", B=1, n=640, H=2, Hk=2, d=128, block_q=64,
                   block_k=128, run=40, clusters=5, alpha=3.0), 0.05),
    (inputs.custom("mixed_n700_d64_q128k64_gqa", B=2, n=700, H=4, Hk=2, d=64, block_q=128,
                   block_k=64, run=40, clusters=5, alpha=3.0), 0.05),
    # 64-row query tiles with an odd T_r: the last 128-row MMA tile reaches 64
    # rows past the statistics' rows
    (inputs.custom("mixed_n130_d128_q64k128", B=2, n=130, H=2, Hk=1, d=128, block_q=64,
                   block_k=128, run=16, clusters=3, alpha=2.0), 0.1),
    (inputs.custom("ragged_n300_d128_t128", B=1, n=300, H=3, Hk=1, d=128, run=16,
                   clusters=4, alpha=2.0), 0.02),
    (inputs.WORKLOADS["clustered_n4096_d64"], 0.05),
    # degenerate shapes: one partial tile per sequence (three sequences), and
    # one full plus one single-row tile
    (inputs.custom("edge_n100_d128_b3", B=3, n=100, H=2, Hk=1, d=128, run=16, clusters=3,
                   alpha=2.0), 0.05),
    (inputs.custom("edge_n65_d64_t64", B=1, n=65, H=1, Hk=1, d=64, block_q=64, block_k=64,
                   run=8, clusters=3, alpha=2.0), 0.3),
]


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__ as g
    g.build()


def _ids(c):
    return f"{c[0].name}-negl{c[1]}"


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_hot_path_matches_oracle(case):
    w, negl = case
    from block_sparse_attention_fwd_gb300 import _lib
    q, k, v, go = inputs.generate(w, seed=0)
    scale = w.scale
    shape = _lib.make_shape(w.B, w.n, w.H, w.Hk, w.d, w.block_q, w.block_k, w.causal, w.window)

    # ---- forward + statistics
    qd, kd, vd, o, lse, stats = U.gpu_forward(shape, q, k, v, scale)
    O, L, S = U.oracle_forward(q, k, v, scale, w.block_q, w.block_k)
    assert U.rel_l2(U.cpu(o), O) <= U.REL_L2
    assert np.abs(U.cpu(lse) - L).max() <= U.LSE_ABS
    err, nchk, small_ok = U.compare_stats(U.cpu(stats), S, L, w.n)
    assert nchk > 0 and err <= U.STATS_ABS and small_ok, (err, small_ok)
    # rows past n hold -inf
    pad = U.cpu(stats)[..., w.n:]
    assert pad.size == 0 or np.all(pad == -np.inf)

    # ---- mask: bit-exact given the GPU's own statistics
    lists = U.gpu_mask(shape, stats, lse, negl)
    ref_on_gpu_stats = U.oracle_mask(U.cpu(stats), U.cpu(lse), w.n, w.block_q, w.block_k, negl)
    U.assert_lists_equal(lists, ref_on_gpu_stats)
    own = U.oracle_mask(S, L, w.n, w.block_q, w.block_k, negl)
    agree = float((U.cpu(lists["mask"]) == own["mask"]).mean())
    assert agree >= 0.999, agree
    if negl == 0.0:
        assert np.all(own["mask"] == 1)

    # ---- backward alone: the oracle's O (as stored), LSE and mask on both sides
    Ob = A.as_stored_output(O)
    o_or = U.to_device_like(Ob, o)
    lse_or = U.to_device_like(L, lse)
    ol = U.lists_to_device(own)
    gq, gk, gv, status = U.gpu_backward(shape, qd, kd, vd, o_or, go, lse_or, scale, ol)
    assert status == 0
    rq, rk, rv = A.backward(q, k, v, Ob, go, L, scale, own["mask"], w.block_q, w.block_k)
    for name, a, b in (("G_Q", gq, rq), ("G_K", gk, rk), ("G_V", gv, rv)):
        e = U.rel_l2(U.cpu(a), b)
        assert e <= U.REL_L2, (name, e)

    # ---- dense backward (lists = NULL), same inputs
    dq2, dk2, dv2, status = U.gpu_backward(shape, qd, kd, vd, o_or, go, lse_or, scale, None)
    assert status == 0
    dq, dk, dv = A.backward(q, k, v, Ob, go, L, scale)
    for name, a, b in (("G_Q", dq2, dq), ("G_K", dk2, dk), ("G_V", dv2, dv)):
        e = U.rel_l2(U.cpu(a), b)
        assert e <= U.REL_L2, (name, e)
    if negl == 0.0:
        # negl_prob = 0 keeps every tile: the listed backward is the dense one.
        # G_K and G_V are accumulated in a fixed order and match bit for bit;
        # G_Q sums fp32 atomic adds whose order varies from run to run.
        assert torch.equal(gk, dk2) and torch.equal(gv, dv2)
        assert U.rel_l2(U.cpu(gq), U.cpu(dq2)) <= 1e-3

    # ---- the whole GPU chain (its own O, LSE and lists) against the oracle's
    # masked backward on the same O, LSE and mask (the forward outputs were
    # checked against the oracle's above, the mask bit for bit)
    cq, ck, cv, status = U.gpu_backward(shape, qd, kd, vd, o, go, lse, scale, lists)
    assert status == 0
    gm = U.cpu(lists["mask"])
    sq, sk, sv = A.backward(q, k, v, U.cpu(o), go, U.cpu(lse), scale, gm, w.block_q, w.block_k)
    for name, a, b in (("G_Q", cq, sq), ("G_K", ck, sk), ("G_V", cv, sv)):
        e = U.rel_l2(U.cpu(a), b)
        assert e <= U.REL_L2, (name, e)


def test_gpu_mask_on_planted_statistics():
    """Hand-built statistics with exact ties, -inf tiles and a NaN tile."""
    from block_sparse_attention_fwd_gb300 import _lib
    B, H, n, b = 1, 2, 256, 64
    shape = _lib.make_shape(B, n, H, H, 64, b, b)
    rng = np.random.default_rng(7)
    T = n // b
    st = np.log(rng.dirichlet(np.full(T, 0.3), size=(B, H, n)).astype(np.float64))
    st = np.transpose(st, (0, 1, 3, 2)).astype(np.float32).copy()   # [B,H,T_c,n]
    st[0, 0, 1, :] = st[0, 0, 0, :]                                  # ties
    st[0, 1, 2, :] = -np.inf                                         # empty tile
    st[0, 1, 3, 5] = np.nan                                          # NaN weight
    lse = np.zeros((B, H, n), dtype=np.float32)
    for negl in (0.0, 0.01, 0.3, 0.9):
        lists = _lib.alloc_lists(shape, "cuda")
        _lib.mask_from_stats(shape, torch.from_numpy(st).cuda(), torch.from_numpy(lse).cuda(),
                             negl, lists)
        ref = U.oracle_mask(st, lse, n, b, b, negl)
        U.assert_lists_equal(lists, ref)
        assert int(lists["nan_count"].item()) == ref["nan_count"] == 1


@pytest.mark.parametrize("tile,d", [(64, 64), (128, 128), (128, 64)])
def test_corrupt_list_entry_is_reported_not_faulted(tile, d):
    from block_sparse_attention_fwd_gb300 import _lib
    w = inputs.custom("corrupt", B=1, n=4 * tile, H=1, Hk=1, d=d, block_q=tile, block_k=tile)
    q, k, v, go = inputs.generate(w)
    shape = _lib.make_shape(w.B, w.n, w.H, w.Hk, w.d, w.block_q, w.block_k, w.causal, w.window)
    qd, kd, vd, o, lse, stats = U.gpu_forward(shape, q, k, v, w.scale)
    lists = U.gpu_mask(shape, stats, lse, 0.05)
    lists["q_idx"][0, 0, 0, 0] = 99          # out of range: T_r = 4
    _, _, _, status = U.gpu_backward(shape, qd, kd, vd, o, go, lse, w.scale, lists)
    assert status == 5                       # BL_ERR_CORRUPT_LISTS
    lists["q_cnt"][0, 0, 1] = 1000
    _, _, _, status = U.gpu_backward(shape, qd, kd, vd, o, go, lse, w.scale, lists)
    assert status == 5


def test_autograd_module_runs_the_chain():
    from block_sparse_attention_fwd_gb300 import BLAttention, _lib
    w = inputs.custom("module", B=1, n=512, H=2, Hk=1, d=64, run=32, clusters=4)
    q, k, v, go = inputs.generate(w)
    qd, kd, vd = (x.cuda().requires_grad_(True) for x in (q, k, v))
    shape = _lib.make_shape(w.B, w.n, w.H, w.Hk, w.d, 128, 128)
    T_r, T_c = _lib.tiles(shape)
    stats = torch.empty((w.B, w.H, T_c, T_r * 128), dtype=torch.float32, device="cuda")
    attn = BLAttention(negl_prob=0.05)
    out, lse = attn(qd, kd, vd, return_softmax_lse=True, tile_stats=stats)
    out.backward(go.cuda())
    O, L, S = A.forward(q, k, v, w.scale, block_q=128, block_k=128)
    assert U.rel_l2(U.cpu(out), O) <= U.REL_L2
    assert np.abs(U.cpu(lse) - L).max() <= U.LSE_ABS
    # the module's mask is the selection rule applied to its own statistics;
    # its gradients against the oracle's backward on its own O, LSE and mask
    gm = U.oracle_mask(U.cpu(stats), U.cpu(lse), w.n, 128, 128, 0.05)["mask"]
    own = U.oracle_mask(S, L, w.n, 128, 128, 0.05)["mask"]
    assert float((gm == own).mean()) >= 0.999
    rq, rk, rv = A.backward(q, k, v, U.cpu(out.detach()), go, U.cpu(lse), w.scale, gm, 128, 128)
    for name, a, b in (("G_Q", qd.grad, rq), ("G_K", kd.grad, rk), ("G_V", vd.grad, rv)):
        e = U.rel_l2(U.cpu(a), b)
        assert e <= U.REL_L2, (name, e)


def test_autograd_module_tile_weights_path():
    """Without a statistics buffer the module's forward keeps only the tile
    weights; its mask is the selection rule on the statistics the forward
    would have written, so its gradients match the oracle's backward under
    the mask of the statistics path on the same inputs."""
    from block_sparse_attention_fwd_gb300 import BLAttention, _lib
    w = inputs.custom("module_tw", B=1, n=1100, H=4, Hk=2, d=128, run=128, clusters=4)
    q, k, v, go = inputs.generate(w)
    shape = _lib.make_shape(w.B, w.n, w.H, w.Hk, w.d, 128, 128)
    assert _lib.fwd_tile_weights_supported(shape)
    T_r, T_c = _lib.tiles(shape)
    attn = BLAttention(negl_prob=0.05)
    stats = torch.empty((w.B, w.H, T_c, T_r * 128), dtype=torch.float32, device="cuda")
    qs, ks, vs = (x.cuda().requires_grad_(True) for x in (q, k, v))
    out_s, lse_s = attn(qs, ks, vs, return_softmax_lse=True, tile_stats=stats)
    gm = U.oracle_mask(U.cpu(stats), U.cpu(lse_s), w.n, 128, 128, 0.05)["mask"]
    assert 0 < float(gm.mean()) < 1
    qd, kd, vd = (x.cuda().requires_grad_(True) for x in (q, k, v))
    out, lse = attn(qd, kd, vd, return_softmax_lse=True)
    out.backward(go.cuda())
    assert torch.equal(out.detach(), out_s.detach())
    assert torch.equal(lse, lse_s)
    rq, rk, rv = A.backward(q, k, v, U.cpu(out.detach()), go, U.cpu(lse), w.scale, gm, 128, 128)
    for name, a, b in (("G_Q", qd.grad, rq), ("G_K", kd.grad, rk), ("G_V", vd.grad, rv)):
        e = U.rel_l2(U.cpu(a), b)
        assert e <= U.REL_L2, (name, e)
