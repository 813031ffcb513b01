"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times, checked against the oracle on sampled heads and tiles.

For every sampled head the oracle computes its own forward, statistics and
mask from the same seeded inputs; the GPU backward is then given the
oracle's lists for those heads (its own lists elsewhere), so both sides
compute the masked gradients of the same mask.  The mask itself is checked
bit for bit by applying the oracle's rule to the GPU's statistics.

The long-context case (n = 131072) checks sampled query tiles against the
oracle (forward rows, statistics, mask rows, G_Q), sampled key tiles of two
whole GQA groups (G_K, G_V) element by element, and, at full size, a
property that holds at any size: the gradients are linear in the mask, so
the sparse gradients plus those of the complementary mask equal the dense
gradients.
"""
import numpy as np
import pytest
import torch

from block_sparse_attention_fwd_gb300 import inputs
from oracle import attention as A
from oracle import mask_spec as M
from tests import parity_util as U

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__ as g
    g.build()
    yield
    torch.cuda.empty_cache()


def _head(x, b, h):
    return x[b, :, h].double().numpy()


def _oracle_head(w, q, k, v, go, b, h):
    hk = h // (w.H // w.Hk)
    qh, kh, vh = _head(q, b, h), _head(k, b, hk), _head(v, b, hk)
    O, L, S = A.forward_head(qh, kh, vh, w.scale, block_k=w.block_k)
    st = np.full((w.T_c, w.T_r * w.block_q), -np.inf)
    st[:, :w.n] = S
    return {"q": qh, "k": kh, "v": vh, "go": _head(go, b, h), "O": O, "L": L, "S": st}


def _oracle_mask_head(w, orc, negl):
    d = M.tile_weights(orc["S"].astype(np.float32), orc["L"].astype(np.float32), w.n, w.block_q)
    T = M.threshold(negl)
    return np.stack([M.select_row(d[i], T)[0] for i in range(w.T_r)])


def _gpu_forward(w, q, k, v):
    from block_sparse_attention_fwd_gb300 import _lib
    shape = _lib.make_shape(w.B, w.n, w.H, w.Hk, w.d, w.block_q, w.block_k, w.causal, w.window)
    return (shape,) + U.gpu_forward(shape, q, k, v, w.scale)


def _check_forward_head(w, o, lse, stats, b, h, orc):
    assert U.rel_l2(U.cpu(o[b, :, h]), orc["O"]) <= U.REL_L2
    assert np.abs(U.cpu(lse[b, h]) - orc["L"]).max() <= U.LSE_ABS
    err, nchk, small_ok = U.compare_stats(U.cpu(stats[b, h])[None, None], orc["S"][None, None],
                                          orc["L"][None, None], w.n)
    assert nchk > 0 and err <= U.STATS_ABS and small_ok, (err, small_ok)


def _check_mask_head(w, stats, lse, lists, b, h, negl, own):
    gst = U.cpu(stats[b, h])
    gl = U.cpu(lse[b, h])
    ref = M.mask_from_stats(gst[None, None], gl[None, None], w.n, w.block_q, w.block_k, negl)
    for key in ("mask", "kv_idx", "kv_cnt", "q_idx", "q_cnt"):
        assert np.array_equal(U.cpu(lists[key][b, h]), ref[key][0, 0]), key
    agree = float((U.cpu(lists["mask"][b, h]) == own).mean())
    assert agree >= 0.995, agree


def _inject_forward(o, lse, b, h, orc, rows=None):
    """Give the backward the oracle's forward results (O as stored, LSE) for
    head h, so that the backward is compared on identical inputs."""
    if rows is None:
        o[b, :, h] = U.to_device_like(A.as_stored_output(orc["O"]), o[b, :, h])
        lse[b, h] = U.to_device_like(orc["L"], lse[b, h])
    else:
        r = torch.as_tensor(rows, device=o.device)
        o[b, r, h] = U.to_device_like(A.as_stored_output(orc["O"]), o[b, r, h])
        lse[b, h, r] = U.to_device_like(orc["L"], lse[b, h, r])


def _inject(lists, b, h, own_mask):
    """Replace head h's lists by the compaction of the oracle's mask."""
    L = M.lists_from_mask(own_mask[None, None])
    for key in ("mask", "kv_idx", "kv_cnt", "q_idx", "q_cnt"):
        lists[key][b, h] = torch.from_numpy(L[key][0, 0]).to(lists[key].device)


# --------------------------------------------------------------- GQA n = 8192
@pytest.fixture(scope="module")
def gqa_case():
    w = inputs.WORKLOADS["gqa_n8192_d128"]
    q, k, v, go = inputs.generate(w, seed=0)
    shape, qd, kd, vd, o, lse, stats = _gpu_forward(w, q, k, v)
    heads = [4, 5, 6, 7]                              # the whole group of kv head 1
    orc = {h: _oracle_head(w, q, k, v, go, 0, h) for h in heads}
    return w, (q, k, v, go), (shape, qd, kd, vd, o, lse, stats), heads, orc


def test_gqa_n8192_forward(gqa_case):
    w, _, (shape, qd, kd, vd, o, lse, stats), heads, orc = gqa_case
    for h in heads:
        _check_forward_head(w, o, lse, stats, 0, h, orc[h])


@pytest.mark.parametrize("negl", [0.01, 0.05, 0.1])
def test_gqa_n8192_mask_and_backward(gqa_case, negl):
    w, (q, k, v, go), (shape, qd, kd, vd, o, lse, stats), heads, orc = gqa_case
    lists = U.gpu_mask(shape, stats, lse, negl)
    own = {h: _oracle_mask_head(w, orc[h], negl) for h in heads}
    o_in, lse_in = o.clone(), lse.clone()
    for h in heads:
        _check_mask_head(w, stats, lse, lists, 0, h, negl, own[h])
        _inject(lists, 0, h, own[h])
        _inject_forward(o_in, lse_in, 0, h, orc[h])
    gq, gk, gv, status = U.gpu_backward(shape, qd, kd, vd, o_in, go, lse_in, w.scale, lists)
    assert status == 0
    hk = heads[0] // (w.H // w.Hk)
    rk = np.zeros((w.n, w.d))
    rv = np.zeros((w.n, w.d))
    for h in heads:
        c = orc[h]
        a, bk, bv = A.backward_head(c["q"], c["k"], c["v"], A.as_stored_output(c["O"]), c["go"],
                                    c["L"], w.scale, own[h], w.block_q, w.block_k)
        assert U.rel_l2(U.cpu(gq[0, :, h]), a) <= U.REL_L2, ("G_Q", h)
        rk += bk
        rv += bv
    assert U.rel_l2(U.cpu(gk[0, :, hk]), rk) <= U.REL_L2
    assert U.rel_l2(U.cpu(gv[0, :, hk]), rv) <= U.REL_L2


# ------------------------------------------------------- video n = 32760 (bench)
def test_video_n32760_sampled_heads():
    w = inputs.WORKLOADS["video_n32760_d128"]
    negl = 0.05
    q, k, v, go = inputs.generate(w, seed=0)
    shape, qd, kd, vd, o, lse, stats = _gpu_forward(w, q, k, v)
    lists = U.gpu_mask(shape, stats, lse, negl)
    heads = [0, 13, 27, 39]
    orc, own = {}, {}
    for h in heads:
        orc[h] = _oracle_head(w, q, k, v, go, 0, h)
        _check_forward_head(w, o, lse, stats, 0, h, orc[h])
        own[h] = _oracle_mask_head(w, orc[h], negl)
        _check_mask_head(w, stats, lse, lists, 0, h, negl, own[h])
        _inject(lists, 0, h, own[h])
    o_in, lse_in = o.clone(), lse.clone()
    for h in heads:
        _inject_forward(o_in, lse_in, 0, h, orc[h])
    gq, gk, gv, status = U.gpu_backward(shape, qd, kd, vd, o_in, go, lse_in, w.scale, lists)
    assert status == 0
    last = w.T_r - 1                                  # ragged: 120 rows / keys
    for h in heads:
        c = orc[h]
        Ob = A.as_stored_output(c["O"])
        for t in (0, 77, 190, last):
            rows = np.arange(t * 128, min(w.n, (t + 1) * 128))
            a, _, _ = A.backward_head(c["q"], c["k"], c["v"], Ob, c["go"], c["L"], w.scale,
                                      own[h], 128, 128, rows=rows)
            assert U.rel_l2(U.cpu(gq[0, rows, h]), a) <= U.REL_L2, ("G_Q", h, t)
            _, bk, bv = A.backward_head(c["q"], c["k"], c["v"], Ob, c["go"], c["L"], w.scale,
                                        own[h], 128, 128, cols=rows)
            if np.linalg.norm(bv) > 0:
                assert U.rel_l2(U.cpu(gk[0, rows, h]), bk) <= U.REL_L2, ("G_K", h, t)
                assert U.rel_l2(U.cpu(gv[0, rows, h]), bv) <= U.REL_L2, ("G_V", h, t)
            else:                                     # no query tile kept this key tile
                assert float(gk[0, rows, h].abs().max()) == 0.0
                assert float(gv[0, rows, h].abs().max()) == 0.0


# ---------------------------------------------------- long context n = 131072
def test_long_n131072_sampled_rows_and_mask_linearity():
    from block_sparse_attention_fwd_gb300 import _lib
    w = inputs.WORKLOADS["long_n131072_d128"]
    negl = 0.05
    q, k, v, go = inputs.generate(w, seed=0)
    shape, qd, kd, vd, o, lse, stats = _gpu_forward(w, q, k, v)
    lists = U.gpu_mask(shape, stats, lse, negl)
    mask = U.cpu(lists["mask"]).copy()
    samples = [(3, 0), (3, 511), (22, 1023), (22, 640)]   # (head, query tile)
    rows_of = {}
    for h, t in samples:
        hk = h // (w.H // w.Hk)
        rows = np.arange(t * 128, (t + 1) * 128)
        qh, kh, vh = _head(q, 0, h), _head(k, 0, hk), _head(v, 0, hk)
        O, L, S = A.forward_head(qh, kh, vh, w.scale, rows=rows, block_k=128)
        assert U.rel_l2(U.cpu(o[0, rows, h]), O) <= U.REL_L2
        assert np.abs(U.cpu(lse[0, h, rows]) - L).max() <= U.LSE_ABS
        gst = U.cpu(stats[0, h, :, rows])                                   # [T_c, 128]
        err, nchk, ok = U.compare_stats(gst[None, None], S[None, None], L[None, None], 128)
        assert nchk > 0 and err <= U.STATS_ABS and ok
        # mask row: bit-exact on the GPU's statistics, and the oracle's own row
        gd = M.tile_weights(gst, U.cpu(lse[0, h, rows]), 128, 128)
        assert np.array_equal(M.select_row(gd[0], M.threshold(negl))[0], mask[0, h, t])
        od = M.tile_weights(S.astype(np.float32), L.astype(np.float32), 128, 128)
        own_row = M.select_row(od[0], M.threshold(negl))[0]
        assert float((own_row == mask[0, h, t]).mean()) >= 0.99
        mask[0, h, t] = own_row
        rows_of[(h, t)] = (rows, qh, kh, vh, O, L)
    # the GPU backward on the mask with the oracle's rows injected, and the
    # oracle's O and LSE for the sampled rows
    o_in, lse_in = o.clone(), lse.clone()
    for (h, t), (rows, qh, kh, vh, O, L) in rows_of.items():
        _inject_forward(o_in, lse_in, 0, h, {"O": O, "L": L}, rows=rows)
    L_all = M.lists_from_mask(mask)
    dev_lists = U.lists_to_device(L_all)
    gq, gk, gv, status = U.gpu_backward(shape, qd, kd, vd, o_in, go, lse_in, w.scale, dev_lists)
    assert status == 0
    for (h, t), (rows, qh, kh, vh, O, L) in rows_of.items():
        # G_Q of these rows needs D and LSE of these rows only
        o_full = np.zeros_like(qh)
        o_full[rows] = A.as_stored_output(O)
        l_full = np.zeros(w.n)
        l_full[rows] = L
        a, _, _ = A.backward_head(qh, kh, vh, o_full, _head(go, 0, h), l_full, w.scale,
                                  mask[0, h], 128, 128, rows=rows)
        assert U.rel_l2(U.cpu(gq[0, rows, h]), a) <= U.REL_L2, ("G_Q", h, t)
    # key-side gradients: G(M) + G(1 - M) = G(dense) at full size
    comp = U.lists_to_device(M.lists_from_mask(1 - mask))
    cq, ck, cv, status = U.gpu_backward(shape, qd, kd, vd, o_in, go, lse_in, w.scale, comp)
    assert status == 0
    dq, dk, dv, status = U.gpu_backward(shape, qd, kd, vd, o_in, go, lse_in, w.scale, None)
    assert status == 0
    for a, c, d in ((gk, ck, dk), (gv, cv, dv), (gq, cq, dq)):
        s = a.float() + c.float()
        e = float((s - d.float()).norm() / d.float().norm())
        assert e <= U.REL_L2, e
    del cq, ck, cv, dq, dk, dv, comp
    # key-side gradients element by element against the oracle: sampled key
    # tiles of two kv heads, each summed over its whole GQA group, from the
    # same O, LSE and mask the GPU backward was given (its forward outputs,
    # validated on the sampled rows above, with the oracle's rows injected)
    G = w.H // w.Hk
    key_tiles = (0, 333, 700, w.T_c - 1)
    cols = np.concatenate([np.arange(j * 128, min(w.n, (j + 1) * 128)) for j in key_tiles])
    for hk in (0, 5):
        kh, vh = _head(k, 0, hk), _head(v, 0, hk)
        rk = np.zeros((len(cols), w.d))
        rv = np.zeros((len(cols), w.d))
        for h in range(hk * G, (hk + 1) * G):
            oh = o_in[0, :, h].float().cpu().double().numpy()
            lh = lse_in[0, h].cpu().double().numpy()
            _, bk, bv = A.backward_head(_head(q, 0, h), kh, vh, oh, _head(go, 0, h), lh, w.scale,
                                        mask[0, h], 128, 128, cols=cols)
            rk += bk
            rv += bv
        for t, j in enumerate(key_tiles):
            sl = slice(t * 128, t * 128 + 128)
            rows = cols[sl]
            if np.linalg.norm(rv[sl]) == 0:           # no query tile kept this key tile
                assert float(gk[0, rows, hk].abs().max()) == 0.0
                assert float(gv[0, rows, hk].abs().max()) == 0.0
                continue
            assert U.rel_l2(U.cpu(gk[0, rows, hk]), rk[sl]) <= U.REL_L2, ("G_K", hk, j)
            assert U.rel_l2(U.cpu(gv[0, rows, hk]), rv[sl]) <= U.REL_L2, ("G_V", hk, j)
    del stats, lists, dev_lists
    _ = _lib
