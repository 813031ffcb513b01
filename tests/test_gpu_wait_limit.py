"""The bounded device-side waits, made to run out on purpose (a limit of 0:
any wait whose phase is not complete at once gives up).  The forward marks
the LSE rows it could not finish with NaN, the backward reports
BL_ERR_TIMEOUT in its status word; both wait for the copies and MMAs they
already issued before freeing their tensor memory, so the next call on the
same GPU runs normally and matches the oracle.  Nothing here faults or hangs
the GPU: every wait is bounded and the failure is only a status."""
import numpy as np
import pytest
import torch

from block_sparse_attention_fwd_gb300 import inputs
from oracle import attention as A
from tests import parity_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__ as g
    g.build()


@pytest.mark.parametrize("tile,d", [(128, 128), (64, 64)])
def test_waits_that_run_out_are_reported_and_the_gpu_stays_usable(tile, d):
    from block_sparse_attention_fwd_gb300 import _lib
    w = inputs.custom("waits", B=1, n=700, H=4, Hk=2, d=d, block_q=tile, block_k=tile, run=40,
                      clusters=6, alpha=3.0)
    q, k, v, go = inputs.generate(w, seed=2)
    shape = _lib.make_shape(w.B, w.n, w.H, w.Hk, w.d, w.block_q, w.block_k)
    # a normal forward and mask, so that the backward below has valid inputs
    qd, kd, vd, o, lse, stats = U.gpu_forward(shape, q, k, v, w.scale)
    lists = U.gpu_mask(shape, stats, lse, 0.05)
    torch.cuda.synchronize()

    prev = _lib.set_wait_limit(0.0)
    try:
        assert prev == pytest.approx(2.0)
        o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
        _lib.attn_fwd(shape, qd, kd, vd, w.scale, o2, lse2, None)
        gq, gk, gv, status = U.gpu_backward(shape, qd, kd, vd, o, go, lse, w.scale, lists)
        torch.cuda.synchronize()
    finally:
        assert _lib.set_wait_limit(-1.0) == 0.0      # back to the default
    assert bool(torch.isnan(lse2).any())            # rows the forward could not finish
    assert status == 6                              # BL_ERR_TIMEOUT

    # the same GPU, normal limit: the whole chain matches the oracle again
    qd, kd, vd, o, lse, stats = U.gpu_forward(shape, q, k, v, w.scale)
    assert not bool(torch.isnan(lse).any())
    lists = U.gpu_mask(shape, stats, lse, 0.05)
    gq, gk, gv, status = U.gpu_backward(shape, qd, kd, vd, o, go, lse, w.scale, lists)
    assert status == 0
    O, L, _ = A.forward(q, k, v, w.scale, block_q=tile, block_k=tile)
    assert U.rel_l2(U.cpu(o), O) <= U.REL_L2
    assert np.abs(U.cpu(lse) - L).max() <= U.LSE_ABS
    ref = A.backward(q, k, v, U.cpu(o), go, U.cpu(lse), w.scale, U.cpu(lists["mask"]), tile, tile)
    for a, b in zip((gq, gk, gv), ref):
        assert U.rel_l2(U.cpu(a), b) <= U.REL_L2
