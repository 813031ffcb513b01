"""The backward reads a work item's lists from global memory, not from its
shared-memory copy, when the GQA group holds more than 32 query heads or
the group's kept entries exceed the copy's capacity (1536).  Both cases,
against the oracle and against the dense backward."""
import numpy as np
import pytest
import torch

from block_sparse_attention_fwd_gb300 import inputs
from oracle import attention as A
from oracle import mask_spec as M
from tests import parity_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__ as g
    g.build()


@pytest.mark.parametrize("d", [64, 128])
def test_group_of_36_heads_matches_oracle(d):
    """H = 36 query heads on one kv head: more heads than the list copy holds."""
    from block_sparse_attention_fwd_gb300 import _lib
    w = inputs.custom("gqa36", B=1, n=700, H=36, Hk=1, d=d, run=128, clusters=5)
    q, k, v, go = inputs.generate(w, seed=5)
    shape = _lib.make_shape(w.B, w.n, w.H, w.Hk, w.d, 128, 128)
    O, L, S = A.forward(q, k, v, w.scale, 128, 128)
    own = M.mask_from_stats(S, L, w.n, 128, 128, 0.05)
    assert 0 < own["mask"].sum() < own["mask"].size
    Ob = A.as_stored_output(O)
    dev = torch.device("cuda")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    o_or = torch.from_numpy(np.ascontiguousarray(Ob)).to(torch.bfloat16).to(dev)
    lse_or = torch.from_numpy(np.ascontiguousarray(L)).float().to(dev)
    gq, gk, gv, status = U.gpu_backward(shape, qd, kd, vd, o_or, go, lse_or, w.scale,
                                        U.lists_to_device(own))
    assert status == 0
    rq, rk, rv = A.backward(q, k, v, Ob, go, L, w.scale, own["mask"], 128, 128)
    for name, a, b in (("G_Q", gq, rq), ("G_K", gk, rk), ("G_V", gv, rv)):
        e = U.rel_l2(U.cpu(a), b)
        assert e <= U.REL_L2, (name, e)


def test_lists_longer_than_the_copy_equal_the_dense_backward():
    """16 query heads x 100 query tiles all kept: 1600 entries per item, more
    than the shared-memory copy holds.  With every tile listed the backward
    is the dense one: dK and dV bit for bit, dQ up to the order of its
    reduce-adds."""
    from block_sparse_attention_fwd_gb300 import _lib
    w = inputs.custom("long_lists", B=1, n=12800, H=16, Hk=1, d=64, run=64, clusters=16)
    q, k, v, go = (x.cuda() for x in inputs.generate(w, seed=6))
    shape = _lib.make_shape(w.B, w.n, w.H, w.Hk, w.d, 128, 128)
    T_r, T_c = _lib.tiles(shape)
    o = torch.empty_like(q)
    lse = torch.empty((1, w.H, w.n), dtype=torch.float32, device="cuda")
    stats = torch.empty((1, w.H, T_c, T_r * 128), dtype=torch.float32, device="cuda")
    _lib.attn_fwd(shape, q, k, v, w.scale, o, lse, stats)
    lists = _lib.alloc_lists(shape, "cuda")
    _lib.mask_from_stats(shape, stats, lse, 0.0, lists)          # negl 0 keeps every tile
    assert int(lists["q_cnt"].sum()) == w.H * T_r * T_c
    listed = U.gpu_backward(shape, q, k, v, o, go, lse, w.scale, lists)
    dense = U.gpu_backward(shape, q, k, v, o, go, lse, w.scale, None)
    assert listed[3] == 0 and dense[3] == 0
    assert torch.equal(listed[1], dense[1]) and torch.equal(listed[2], dense[2])
    assert U.rel_l2(U.cpu(listed[0]), U.cpu(dense[0])) <= 1e-3
