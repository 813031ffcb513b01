"""bl_attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (a host runtime that owns all device memory through its own pool, or
a caller that cannot accept cudaMalloc's implicit synchronisation).  It uses
the library's fixed device scratch array instead of a caller workspace.

Collected last on purpose (file name), so a run that stops at the first
failure has already run every other test.  Runs alone in a fresh process as
well as after the other tests.
"""
import ctypes

import pytest
import torch

from block_sparse_attention_fwd_gb300 import inputs

REL_L2 = 1e-2    # the tolerance of the parity tests


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm().clamp_min(1e-30))


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """No GPU needed: the size check runs on the host before any launch."""
    import __graft_entry__ as g
    g.build()
    from block_sparse_attention_fwd_gb300 import _lib
    lib = _lib.load()
    big = _lib.make_shape(1, 65536, 8, 8, 128, 128, 128)      # needs ~270 MB of scratch
    assert _lib.bwd_workspace_bytes(big) > 32 * 1024 * 1024
    fake = ctypes.c_void_p(0x10000)
    r = lib.bl_attn_bwd_noalloc(ctypes.byref(big), fake, fake, fake, fake, fake, fake, 0.1, None,
                                fake, fake, fake, None)
    assert r == 4                                               # BL_ERR_WORKSPACE
    assert lib.bl_bwd_noalloc_check_status(ctypes.byref(big), None) == 4


def _case(name, n, H, Hk, d, tile, seed):
    from block_sparse_attention_fwd_gb300 import _lib
    w = inputs.custom(name, B=1, n=n, H=H, Hk=Hk, d=d, block_q=tile, block_k=tile,
                      run=40, clusters=6, alpha=3.0)
    q, k, v, go = inputs.generate(w, seed=seed)
    dev = torch.device("cuda")
    shape = _lib.make_shape(w.B, w.n, w.H, w.Hk, w.d, w.block_q, w.block_k, w.causal, w.window)
    assert _lib.bwd_workspace_bytes(shape) <= 32 * 1024 * 1024
    qd, kd, vd, god = (x.to(dev) for x in (q, k, v, go))
    o = torch.empty_like(qd)
    lse = torch.empty((w.B, w.H, w.n), dtype=torch.float32, device=dev)
    T_r, T_c = _lib.tiles(shape)
    stats = torch.empty((w.B, w.H, T_c, T_r * tile), dtype=torch.float32, device=dev)
    _lib.attn_fwd(shape, qd, kd, vd, w.scale, o, lse, stats)
    return w, shape, (q, k, v, go), (qd, kd, vd, god, o, lse, stats)


@pytest.mark.gpu
@pytest.mark.parametrize("tile,d,negl", [(128, 128, 0.05), (64, 64, 0.1)])
def test_noalloc_matches_workspace_backward_and_oracle(tile, d, negl):
    """Two shapes in a row (the larger first, so the second call's scratch
    offsets differ from what the array holds), each called twice: every call
    must match the workspace backward and the oracle, with a clear status."""
    import __graft_entry__ as g
    g.build()
    from block_sparse_attention_fwd_gb300 import _lib
    from oracle import attention as A
    from tests import parity_util as U
    for name, n, H, Hk, seed in (("noalloc_big", 2000, 8, 4, 5), ("noalloc", 1000, 4, 2, 3)):
        w, shape, (q, k, v, go), (qd, kd, vd, god, o, lse, stats) = _case(
            name, n, H, Hk, d, tile, seed)
        dev = qd.device
        lists = _lib.alloc_lists(shape, dev)
        _lib.mask_from_stats(shape, stats, lse, negl, lists)
        ref = [torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)]
        ws = torch.empty(_lib.bwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)
        _lib.attn_bwd(shape, qd, kd, vd, o, god, lse, w.scale, lists, *ref, ws)
        assert _lib.bwd_check_status(shape, ws) == 0
        # the oracle's masked backward on the GPU's own O, LSE and mask
        orc = A.backward(q, k, v, U.cpu(o), go, U.cpu(lse), w.scale, U.cpu(lists["mask"]),
                         tile, tile)
        for _ in range(2):       # the second call must not see the first call's scratch
            out = [torch.full_like(qd, float("nan")), torch.full_like(kd, float("nan")),
                   torch.full_like(vd, float("nan"))]
            _lib.attn_bwd_noalloc(shape, qd, kd, vd, o, god, lse, w.scale, lists, *out)
            assert _lib.bwd_noalloc_check_status(shape) == 0
            for a, b, r in zip(out, ref, orc):
                assert torch.isfinite(a).all()
                assert _rel(a, b) <= REL_L2
                assert U.rel_l2(U.cpu(a), r) <= REL_L2


@pytest.mark.gpu
def test_noalloc_status_reports_a_corrupt_list_entry():
    import __graft_entry__ as g
    g.build()
    from block_sparse_attention_fwd_gb300 import _lib
    w, shape, _, (qd, kd, vd, god, o, lse, stats) = _case("noalloc_corrupt", 512, 2, 1, 128,
                                                          128, 1)
    lists = _lib.alloc_lists(shape, qd.device)
    _lib.mask_from_stats(shape, stats, lse, 0.05, lists)
    out = [torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)]
    _lib.attn_bwd_noalloc(shape, qd, kd, vd, o, god, lse, w.scale, lists, *out)
    assert _lib.bwd_noalloc_check_status(shape) == 0
    bad = {k_: t.clone() for k_, t in lists.items()}
    bad["q_idx"][0, 0, 0, 0] = 99            # out of range: T_r = 4
    _lib.attn_bwd_noalloc(shape, qd, kd, vd, o, god, lse, w.scale, bad, *out)
    assert _lib.bwd_noalloc_check_status(shape) == 5    # BL_ERR_CORRUPT_LISTS
    _lib.attn_bwd_noalloc(shape, qd, kd, vd, o, god, lse, w.scale, lists, *out)
    assert _lib.bwd_noalloc_check_status(shape) == 0    # the next call starts clean
