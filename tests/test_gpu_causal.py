"""GPU parity of causal and causal sliding-window attention ("Introducing
BackLite", Training Nanochat: decoder training with windows of 1024 and
2048) against the fp64 oracle, through the C ABI: forward and tile
statistics, the mask (bit-exact on the GPU's statistics, structurally empty
tiles never kept), and the listed and dense backward."""
import numpy as np
import pytest
import torch

from block_sparse_attention_fwd_gb300 import inputs
from oracle import attention as A
from oracle import mask_spec as M
from tests import parity_util as U

pytestmark = pytest.mark.gpu

CASES = [
    # causal, GQA, ragged tail, T_r odd (last forward pair holds one tile)
    (inputs.custom("causal_n1000_d128_gqa", B=1, n=1000, H=4, Hk=2, d=128, run=48,
                   clusters=8, causal=True), 0.05),
    (inputs.custom("causal_n777_d64", B=2, n=777, H=2, Hk=1, d=64, run=32, clusters=6,
                   alpha=2.5, causal=True), 0.02),
    # windows: not a multiple of the tile, exactly one tile, wider than n
    (inputs.custom("window300_n1200_d128", B=1, n=1200, H=2, Hk=2, d=128, run=40,
                   clusters=5, causal=True, window=300), 0.05),
    (inputs.custom("window128_n640_d64", B=1, n=640, H=2, Hk=1, d=64, run=24, clusters=4,
                   causal=True, window=128), 0.1),
    (inputs.custom("window2048_n900_d128", B=1, n=900, H=1, Hk=1, d=128, run=32,
                   clusters=4, causal=True, window=2048), 0.0),
]


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__ as g
    g.build()


def _ids(c):
    return f"{c[0].name}-negl{c[1]}"


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_causal_hot_path_matches_oracle(case):
    w, negl = case
    from block_sparse_attention_fwd_gb300 import _lib
    q, k, v, go = inputs.generate(w, seed=0)
    scale = w.scale
    shape = _lib.make_shape(w.B, w.n, w.H, w.Hk, w.d, w.block_q, w.block_k, w.causal, w.window)

    qd, kd, vd, o, lse, stats = U.gpu_forward(shape, q, k, v, scale)
    O, L, S = A.forward(q, k, v, scale, w.block_q, w.block_k, causal=w.causal, window=w.window)
    assert U.rel_l2(U.cpu(o), O) <= U.REL_L2
    assert np.abs(U.cpu(lse) - L).max() <= U.LSE_ABS
    err, nchk, small_ok = U.compare_stats(U.cpu(stats), S, L, w.n)
    assert nchk > 0 and err <= U.STATS_ABS and small_ok, (err, small_ok)
    # tiles without an attending pair carry -inf for every row
    st = U.cpu(stats)
    empty = M.structurally_empty(w.T_r, w.T_c, w.n, w.block_q, w.block_k, w.causal, w.window)
    for i, j in np.argwhere(empty):
        assert np.all(st[:, :, j, i * w.block_q:(i + 1) * w.block_q] == -np.inf), (i, j)

    lists = U.gpu_mask(shape, stats, lse, negl)
    ref = M.mask_from_stats(st, U.cpu(lse), w.n, w.block_q, w.block_k, negl,
                            causal=w.causal, window=w.window)
    U.assert_lists_equal(lists, ref)
    own = M.mask_from_stats(S, L, w.n, w.block_q, w.block_k, negl, causal=w.causal,
                            window=w.window)
    assert not np.any(U.cpu(lists["mask"])[:, :, empty])
    if negl == 0.0:
        assert np.array_equal(own["mask"][0, 0], (~empty).astype(np.uint8))

    Ob = A.as_stored_output(O)
    o_or = U.to_device_like(Ob, o)
    lse_or = U.to_device_like(L, lse)
    rq, rk, rv = A.backward(q, k, v, Ob, go, L, scale, own["mask"], w.block_q, w.block_k,
                            causal=w.causal, window=w.window)
    gq, gk, gv, status = U.gpu_backward(shape, qd, kd, vd, o_or, go, lse_or, scale,
                                        U.lists_to_device(own))
    assert status == 0
    for name, a, b in (("G_Q", gq, rq), ("G_K", gk, rk), ("G_V", gv, rv)):
        e = U.rel_l2(U.cpu(a), b)
        assert e <= U.REL_L2, (name, e)


@pytest.mark.parametrize("window", [0, 300])
def test_causal_dense_backward_matches_oracle(window):
    """Without lists the backward visits every structurally non-empty tile and
    masks the diagonal ones: it equals the oracle's exact causal gradient."""
    w = inputs.custom("causal_dense_n700_d128", B=1, n=700, H=2, Hk=1, d=128, run=32,
                      clusters=6, causal=True, window=window)
    from block_sparse_attention_fwd_gb300 import _lib
    q, k, v, go = inputs.generate(w, seed=3)
    scale = w.scale
    shape = _lib.make_shape(w.B, w.n, w.H, w.Hk, w.d, w.block_q, w.block_k, w.causal, w.window)
    O, L, _ = A.forward(q, k, v, scale, w.block_q, w.block_k, causal=True, window=window)
    Ob = A.as_stored_output(O)
    dev = torch.device("cuda")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    o_or = torch.from_numpy(np.ascontiguousarray(Ob)).to(torch.bfloat16).to(dev)
    lse_or = torch.from_numpy(np.ascontiguousarray(L)).float().to(dev)
    gq, gk, gv, status = U.gpu_backward(shape, qd, kd, vd, o_or, go, lse_or, scale, None)
    assert status == 0
    rq, rk, rv = A.backward(q, k, v, Ob, go, L, scale, None, w.block_q, w.block_k,
                            causal=True, window=window)
    for name, a, b in (("G_Q", gq, rq), ("G_K", gk, rk), ("G_V", gv, rv)):
        e = U.rel_l2(U.cpu(a), b)
        assert e <= U.REL_L2, (name, e)


def test_causal_autograd_module_matches_torch():
    """BLAttention(causal, window) with negl 0 against torch SDPA on the GPU."""
    from block_sparse_attention_fwd_gb300.api import BLAttention
    torch.manual_seed(0)
    B, n, H, d, W = 1, 520, 2, 64, 200
    q = torch.randn(B, n, H, d, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    k = torch.randn(B, n, H, d, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    v = torch.randn(B, n, H, d, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    g = torch.randn(B, n, H, d, device="cuda", dtype=torch.bfloat16)
    o = BLAttention(0.0, causal=True, window=W)(q, k, v)
    o.backward(g)
    r = torch.arange(n, device="cuda")
    allow = (r[None, :] <= r[:, None]) & (r[None, :] > r[:, None] - W)
    qf, kf, vf = (x.detach().float().transpose(1, 2).requires_grad_() for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qf, kf, vf, attn_mask=allow)
    ref.backward(g.float().transpose(1, 2))
    assert U.rel_l2(U.cpu(o), ref.detach().transpose(1, 2).cpu().numpy()) <= U.REL_L2
    for a, b in ((q, qf), (k, kf), (v, vf)):
        assert U.rel_l2(U.cpu(a.grad), b.grad.transpose(1, 2).cpu().numpy()) <= U.REL_L2
