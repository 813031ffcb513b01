"""GPU parity of packed variable-length batches through the C ABI
(bl_*_varlen) against the fp64 oracle: forward and tile statistics, the mask
(bit-exact on the GPU's own statistics), and the listed and dense backward.
The packed results must also equal, bit for bit, the fixed-length calls on
each sequence alone: the forward and the mask are deterministic, so any
difference is a slicing or offset error."""
import numpy as np
import pytest
import torch

from block_sparse_attention_fwd_gb300 import inputs
from oracle import attention as A
from oracle import varlen as V
from tests import parity_util as U

pytestmark = pytest.mark.gpu

CASES = [
    # tcgen05 path: ragged tails, length 1, a run of equal lengths (one launch
    # group of B = 3), an empty sequence, GQA
    ("tc_d128_gqa", dict(H=4, Hk=2, d=128, block=128, causal=False, window=0),
     [1, 127, 128, 129, 300, 300, 300, 1000, 0, 64], 0.05),
    # causal sliding window, head dim 64
    ("tc_d64_window200", dict(H=2, Hk=1, d=64, block=128, causal=True, window=200),
     [700, 1, 333, 333, 1500], 0.05),
    # 64 x 64 tiles (mma.sync path)
    ("mma_d64_tile64", dict(H=2, Hk=2, d=64, block=64, causal=False, window=0),
     [200, 64, 65, 500, 0], 0.1),
]


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__ as g
    g.build()


def _setup(cfg, lengths, seed=0, streams=0):
    from block_sparse_attention_fwd_gb300 import _lib
    w = inputs.custom("packed", B=1, n=1, H=cfg["H"], Hk=cfg["Hk"], d=cfg["d"],
                      block_q=cfg["block"], block_k=cfg["block"], run=32, clusters=6,
                      causal=cfg["causal"], window=cfg["window"])
    cu, q, k, v, go = inputs.generate_packed(w, lengths, seed=seed)
    vl = _lib.Varlen(cu, cfg["H"], cfg["Hk"], cfg["d"], cfg["block"], cfg["block"],
                     cfg["causal"], cfg["window"], streams)
    return w, cu, q, k, v, go, vl


def _gpu_forward(vl, q, k, v, scale):
    from block_sparse_attention_fwd_gb300 import _lib
    dev = torch.device("cuda")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty(vl.sizes["lse"], dtype=torch.float32, device=dev)
    stats = torch.empty(vl.sizes["tile_stats"], dtype=torch.float32, device=dev)
    _lib.attn_fwd_varlen(vl, qd, kd, vd, scale, o, lse, stats)
    return qd, kd, vd, o, lse, stats


def _flat_lists_to_device(lists_np):
    out = {key: torch.from_numpy(np.ascontiguousarray(val)).to("cuda")
           for key, val in lists_np.items() if key != "nan_count"}
    out["nan_count"] = torch.zeros(1, dtype=torch.int32, device="cuda")
    return out


@pytest.mark.parametrize("name,cfg,lengths,negl", CASES, ids=[c[0] for c in CASES])
def test_varlen_hot_path_matches_oracle(name, cfg, lengths, negl):
    from block_sparse_attention_fwd_gb300 import _lib
    w, cu, q, k, v, go, vl = _setup(cfg, lengths)
    H, bq, bk = cfg["H"], cfg["block"], cfg["block"]
    causal, window = cfg["causal"], cfg["window"]
    scale = cfg["d"] ** -0.5

    qd, kd, vd, o, lse, stats = _gpu_forward(vl, q, k, v, scale)
    O, L, S = V.forward(q, k, v, cu, scale, bq, bk, causal, window)
    assert U.rel_l2(U.cpu(o), O) <= U.REL_L2
    assert np.abs(U.cpu(lse) - L).max() <= U.LSE_ABS
    seqs, _ = V.layout(cu, H, bq, bk)
    g_st = U.cpu(stats)
    for s in seqs:
        if s["n"] == 0:
            continue
        n, T_r, T_c = s["n"], s["T_r"], s["T_c"]
        size = H * T_c * T_r * bq
        gs = g_st[s["stats"]:s["stats"] + size].reshape(1, H, T_c, -1)
        os_ = S[s["stats"]:s["stats"] + size].reshape(1, H, T_c, -1)
        ls = L[s["lse"]:s["lse"] + H * n].reshape(1, H, n)
        err, nchk, small_ok = U.compare_stats(gs, os_, ls, n)
        assert nchk > 0 and err <= U.STATS_ABS and small_ok, (s["tok"], err, small_ok)

    lists = _lib.alloc_varlen_lists(vl, qd.device)
    _lib.mask_from_stats_varlen(vl, stats, lse, negl, lists)
    ref = V.mask_from_stats(g_st, U.cpu(lse), cu, H, bq, bk, negl, causal, window)
    U.assert_lists_equal(lists, ref)
    assert int(lists["nan_count"].item()) == ref["nan_count"] == 0
    mask = U.cpu(lists["mask"])
    if negl > 0:
        assert 0 < mask.sum() < mask.size

    own = V.mask_from_stats(S, L, cu, H, bq, bk, negl, causal, window)
    Ob = A.as_stored_output(O)
    o_or = U.to_device_like(Ob, o)
    lse_or = U.to_device_like(L, lse)
    god = go.to("cuda")
    ws = torch.empty(vl.sizes["bwd_workspace_bytes"], dtype=torch.uint8, device="cuda")
    for lists_in, m in ((_flat_lists_to_device(own), own["mask"]), (None, None)):
        g_q, g_k, g_v = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        _lib.attn_bwd_varlen(vl, qd, kd, vd, o_or, god, lse_or, scale, lists_in, g_q, g_k, g_v,
                             ws)
        assert _lib.varlen_bwd_check_status(vl, ws) == 0
        rq, rk, rv = V.backward(q, k, v, Ob, go, L, cu, scale, m, bq, bk, causal, window)
        for gname, a, b in (("G_Q", g_q, rq), ("G_K", g_k, rk), ("G_V", g_v, rv)):
            e = U.rel_l2(U.cpu(a), b)
            assert e <= U.REL_L2, (gname, m is None, e)


@pytest.mark.parametrize("name,cfg,lengths,negl", CASES, ids=[c[0] for c in CASES])
def test_varlen_equals_fixed_length_calls_per_sequence(name, cfg, lengths, negl):
    """Forward outputs, statistics and lists of the packed call equal, bit for
    bit, the fixed-length calls (B = 1) on each sequence."""
    from block_sparse_attention_fwd_gb300 import _lib
    w, cu, q, k, v, go, vl = _setup(cfg, lengths, seed=4)
    H, bq = cfg["H"], cfg["block"]
    scale = cfg["d"] ** -0.5
    qd, kd, vd, o, lse, stats = _gpu_forward(vl, q, k, v, scale)
    lists = _lib.alloc_varlen_lists(vl, qd.device)
    _lib.mask_from_stats_varlen(vl, stats, lse, negl, lists)
    seqs, _ = V.layout(cu, H, bq, bq)
    for si, s in enumerate(seqs):
        n = s["n"]
        if n == 0:
            continue
        a = s["tok"]
        shape = vl.seq_shape(si)
        q1, k1, v1 = (x[None, a:a + n] for x in (q, k, v))
        _, _, _, o1, l1, st1 = U.gpu_forward(shape, q1, k1, v1, scale)
        assert torch.equal(o[a:a + n], o1[0])
        assert torch.equal(lse[s["lse"]:s["lse"] + H * n], l1.reshape(-1))
        assert torch.equal(stats[s["stats"]:s["stats"] + st1.numel()], st1.reshape(-1))
        l1s = U.gpu_mask(shape, st1, l1, negl)
        T_r, T_c = s["T_r"], s["T_c"]
        for key, off, size in (("mask", "mask", H * T_r * T_c), ("kv_idx", "mask", H * T_r * T_c),
                               ("kv_cnt", "kv_cnt", H * T_r), ("q_idx", "q_idx", H * T_c * T_r),
                               ("q_cnt", "q_cnt", H * T_c)):
            assert torch.equal(lists[key][s[off]:s[off] + size], l1s[key].reshape(-1)), key


TW_CASES = [c for c in CASES if c[1]["block"] == 128] + [
    # many launch groups on eight side streams, sharing the statistics slots
    ("tc_d128_streams", dict(H=4, Hk=4, d=128, block=128, causal=False, window=0),
     [900, 130, 2000, 1, 640, 640, 256, 1500], 0.05),
]


@pytest.mark.parametrize("name,cfg,lengths,negl", TW_CASES, ids=[c[0] for c in TW_CASES])
def test_varlen_tile_weights_equal_the_statistics_path(name, cfg, lengths, negl):
    """bl_attn_fwd_tile_weights_varlen leaves O, LSE and the statistics as the
    plain packed forward writes them, its tile weights equal the fixed-length
    call's on each sequence (with or without a statistics output), and the
    lists built from them equal the lists built from the statistics, bit for
    bit."""
    from block_sparse_attention_fwd_gb300 import _lib
    w, cu, q, k, v, go, vl = _setup(cfg, lengths, seed=6, streams=8)
    H, bq = cfg["H"], cfg["block"]
    scale = cfg["d"] ** -0.5
    assert _lib.fwd_tile_weights_supported_varlen(vl)
    qd, kd, vd, o, lse, stats = _gpu_forward(vl, q, k, v, scale)
    z = vl.sizes
    o1, lse1, st1 = torch.empty_like(o), torch.empty_like(lse), torch.empty_like(stats)
    lw1 = torch.empty(z["mask"], dtype=torch.float32, device="cuda")
    _lib.attn_fwd_tile_weights_varlen(vl, qd, kd, vd, scale, o1, lse1, lw1, tile_stats=st1)
    o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
    lw2 = torch.full_like(lw1, float("nan"))
    ws = torch.empty(_lib.fwd_workspace_bytes_varlen(vl), dtype=torch.uint8, device="cuda")
    _lib.attn_fwd_tile_weights_varlen(vl, qd, kd, vd, scale, o2, lse2, lw2, workspace=ws)
    torch.cuda.synchronize()
    for a, b in ((o, o1), (o, o2), (lse, lse1), (lse, lse2), (stats, st1)):
        assert torch.equal(a, b)
    assert torch.equal(lw1.view(torch.int32), lw2.view(torch.int32))
    seqs, _ = V.layout(cu, H, bq, bq)
    for si, s in enumerate(seqs):
        n = s["n"]
        if n == 0:
            continue
        a = s["tok"]
        shape = vl.seq_shape(si)
        T_r, T_c = s["T_r"], s["T_c"]
        q1, k1, v1 = (x[None, a:a + n].cuda() for x in (q, k, v))
        oo = torch.empty_like(q1)
        ll = torch.empty((1, H, n), dtype=torch.float32, device="cuda")
        lw = torch.empty((1, H, T_r, T_c), dtype=torch.float32, device="cuda")
        wsf = torch.empty(_lib.fwd_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
        _lib.attn_fwd_tile_weights(shape, q1, k1, v1, scale, oo, ll, lw, workspace=wsf)
        blk = lw2[s["mask"]:s["mask"] + H * T_r * T_c]
        assert torch.equal(blk.view(torch.int32), lw.reshape(-1).view(torch.int32)), si
    for ng in (negl, 0.3):
        la = _lib.alloc_varlen_lists(vl, qd.device)
        _lib.mask_from_tile_weights_varlen(vl, lw2, ng, la)
        lb = _lib.alloc_varlen_lists(vl, qd.device)
        _lib.mask_from_stats_varlen(vl, stats, lse, ng, lb)
        for key in ("mask", "kv_idx", "kv_cnt", "q_idx", "q_cnt"):
            assert torch.equal(la[key], lb[key]), (key, ng)


def test_varlen_corrupt_list_is_reported():
    """An out-of-range q_idx entry in one sequence's block is skipped on the
    device and reported by bl_varlen_bwd_check_status."""
    from block_sparse_attention_fwd_gb300 import _lib
    cfg = dict(H=2, Hk=2, d=128, block=128, causal=False, window=0)
    w, cu, q, k, v, go, vl = _setup(cfg, [300, 200, 200], seed=2)
    scale = 128 ** -0.5
    qd, kd, vd, o, lse, stats = _gpu_forward(vl, q, k, v, scale)
    lists = _lib.alloc_varlen_lists(vl, qd.device)
    _lib.mask_from_stats_varlen(vl, stats, lse, 0.0, lists)
    seqs, _ = V.layout(cu, 2, 128, 128)
    lists["q_idx"][seqs[2]["q_idx"]] = 99          # the last run: sequences 1 and 2
    ws = torch.empty(vl.sizes["bwd_workspace_bytes"], dtype=torch.uint8, device="cuda")
    g = [torch.empty_like(x) for x in (qd, kd, vd)]
    _lib.attn_bwd_varlen(vl, qd, kd, vd, o, go.to("cuda"), lse, scale, lists, *g, ws)
    assert _lib.varlen_bwd_check_status(vl, ws) == 5
    lists["q_idx"][seqs[2]["q_idx"]] = 0
    _lib.attn_bwd_varlen(vl, qd, kd, vd, o, go.to("cuda"), lse, scale, lists, *g, ws)
    assert _lib.varlen_bwd_check_status(vl, ws) == 0


def test_varlen_autograd_module_matches_torch():
    """BLAttention.varlen with negl 0 (dense backward) against torch SDPA over
    the packed axis with a block-diagonal causal mask, on the GPU."""
    from block_sparse_attention_fwd_gb300.api import BLAttention
    torch.manual_seed(1)
    cu = [0, 90, 90, 400, 401, 700]
    T, H, Hk, d = cu[-1], 2, 1, 64
    q = torch.randn(T, H, d, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    k = torch.randn(T, Hk, d, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    v = torch.randn(T, Hk, d, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    g = torch.randn(T, H, d, device="cuda", dtype=torch.bfloat16)
    o = BLAttention(0.0, causal=True).varlen(q, k, v, cu)
    o.backward(g)
    seq = torch.zeros(T, dtype=torch.long, device="cuda")
    for s in range(len(cu) - 1):
        seq[cu[s]:cu[s + 1]] = s
    r = torch.arange(T, device="cuda")
    allow = (seq[:, None] == seq[None, :]) & (r[None, :] <= r[:, None])
    qf = q.detach().float().transpose(0, 1)[None].requires_grad_()
    kf = k.detach().float().repeat_interleave(H // Hk, 1).transpose(0, 1)[None].requires_grad_()
    vf = v.detach().float().repeat_interleave(H // Hk, 1).transpose(0, 1)[None].requires_grad_()
    ref = torch.nn.functional.scaled_dot_product_attention(qf, kf, vf, attn_mask=allow)
    ref.backward(g.float().transpose(0, 1)[None])
    assert U.rel_l2(U.cpu(o), ref.detach()[0].transpose(0, 1).cpu().numpy()) <= U.REL_L2
    assert U.rel_l2(U.cpu(q.grad), qf.grad[0].transpose(0, 1).cpu().numpy()) <= U.REL_L2
    for a, b in ((k, kf), (v, vf)):
        want = b.grad[0].transpose(0, 1).reshape(T, Hk, H // Hk, d).sum(2)
        assert U.rel_l2(U.cpu(a.grad), want.cpu().numpy()) <= U.REL_L2


def test_varlen_concurrent_runs_match_serial_runs():
    """Runs spread over side streams give the same forward, statistics and
    lists, bit for bit, as runs one after another on the caller's stream, and
    the same gradients up to the order of the dQ reduce-adds; a later kernel
    on the caller's stream sees every run's output (the join)."""
    from block_sparse_attention_fwd_gb300 import _lib
    cfg = dict(H=4, Hk=2, d=128, block=128, causal=True, window=0)
    lengths = [900, 130, 2000, 1, 640, 640, 256, 1500]
    res = {}
    for streams in (1, 2, 8):
        w, cu, q, k, v, go, vl = _setup(cfg, lengths, seed=6, streams=streams)
        scale = 128 ** -0.5
        qd, kd, vd, o, lse, stats = _gpu_forward(vl, q, k, v, scale)
        lists = _lib.alloc_varlen_lists(vl, qd.device)
        _lib.mask_from_stats_varlen(vl, stats, lse, 0.05, lists)
        ws = torch.empty(vl.sizes["bwd_workspace_bytes"], dtype=torch.uint8, device="cuda")
        g = [torch.empty_like(x) for x in (qd, kd, vd)]
        _lib.attn_bwd_varlen(vl, qd, kd, vd, o, go.to("cuda"), lse, scale, lists, *g, ws)
        sums = torch.stack([x.float().abs().sum() for x in g])   # on the caller's stream
        assert _lib.varlen_bwd_check_status(vl, ws) == 0
        res[streams] = (o, lse, stats, lists, g, sums)
    o1, l1, s1, li1, g1, sum1 = res[1]
    for streams in (2, 8):
        o, lse, stats, lists, g, sums = res[streams]
        assert torch.equal(o, o1) and torch.equal(lse, l1) and torch.equal(stats, s1)
        for key in ("mask", "kv_idx", "kv_cnt", "q_idx", "q_cnt"):
            assert torch.equal(lists[key], li1[key]), key
        assert torch.equal(g[1], g1[1]) and torch.equal(g[2], g1[2])   # dK, dV: one writer
        assert U.rel_l2(U.cpu(g[0]), U.cpu(g1[0])) <= 1e-3
        assert torch.allclose(sums, sum1, rtol=1e-3)
