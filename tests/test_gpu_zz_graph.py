"""The three calls, fixed-length and packed, captured in a CUDA graph and
replayed: the replay must reproduce the eager results (the forward and the
mask bit for bit; the gradients up to the order of the dQ reduce-adds).
The packed calls fork to the library's side streams and join back, which
stream capture must follow.  The library's side streams are created by an
eager call before the capture."""
import pytest
import torch

from block_sparse_attention_fwd_gb300 import inputs
from tests import parity_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__ as g
    g.build()


def _compare(eager, replay):
    o, lse, stats, mask, g = eager
    o2, lse2, stats2, mask2, g2 = replay
    assert torch.equal(o, o2) and torch.equal(lse, lse2) and torch.equal(stats, stats2)
    assert torch.equal(mask, mask2)
    assert torch.equal(g[1], g2[1]) and torch.equal(g[2], g2[2])
    assert U.rel_l2(U.cpu(g2[0]), U.cpu(g[0])) <= 1e-3


def test_fixed_length_chain_replays_from_a_graph():
    from block_sparse_attention_fwd_gb300 import _lib
    w = inputs.custom("graph", B=1, n=1500, H=4, Hk=2, d=128, run=32, clusters=6)
    q, k, v, go = (x.cuda() for x in inputs.generate(w, seed=1))
    shape = _lib.make_shape(w.B, w.n, w.H, w.Hk, w.d, 128, 128)
    T_r, T_c = _lib.tiles(shape)
    o = torch.empty_like(q)
    lse = torch.empty((1, w.H, w.n), dtype=torch.float32, device="cuda")
    stats = torch.empty((1, w.H, T_c, T_r * 128), dtype=torch.float32, device="cuda")
    lists = _lib.alloc_lists(shape, "cuda")
    g = [torch.empty_like(x) for x in (q, k, v)]
    ws = torch.empty(_lib.bwd_workspace_bytes(shape), dtype=torch.uint8, device="cuda")

    def chain():
        _lib.attn_fwd(shape, q, k, v, w.scale, o, lse, stats)
        _lib.mask_from_stats(shape, stats, lse, 0.05, lists)
        _lib.attn_bwd(shape, q, k, v, o, go, lse, w.scale, lists, *g, ws)

    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        chain()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (o, lse, stats, lists["mask"])] + [[x.clone() for x in g]]
    for t in (o, lse, stats, *g):
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        chain()
    graph.replay()
    torch.cuda.synchronize()
    assert _lib.bwd_check_status(shape, ws) == 0
    _compare(eager, [o, lse, stats, lists["mask"], g])


def test_packed_chain_replays_from_a_graph():
    from block_sparse_attention_fwd_gb300 import _lib
    base = inputs.custom("graph_packed", B=1, n=1, H=4, Hk=2, d=128, run=32, clusters=6,
                         causal=True)
    cu, q, k, v, go = inputs.generate_packed(base, [700, 130, 130, 1, 1200, 0, 450], seed=2)
    q, k, v, go = (x.cuda() for x in (q, k, v, go))
    vl = _lib.Varlen(cu, 4, 2, 128, 128, 128, 1, 0)
    scale = 128 ** -0.5
    o = torch.empty_like(q)
    lse = torch.empty(vl.sizes["lse"], dtype=torch.float32, device="cuda")
    stats = torch.empty(vl.sizes["tile_stats"], dtype=torch.float32, device="cuda")
    lists = _lib.alloc_varlen_lists(vl, "cuda")
    g = [torch.empty_like(x) for x in (q, k, v)]
    ws = torch.empty(vl.sizes["bwd_workspace_bytes"], dtype=torch.uint8, device="cuda")

    def chain():
        _lib.attn_fwd_varlen(vl, q, k, v, scale, o, lse, stats)
        _lib.mask_from_stats_varlen(vl, stats, lse, 0.05, lists)
        _lib.attn_bwd_varlen(vl, q, k, v, o, go, lse, scale, lists, *g, ws)

    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        chain()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (o, lse, stats, lists["mask"])] + [[x.clone() for x in g]]
    for t in (o, lse, stats, *g):
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        chain()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert _lib.varlen_bwd_check_status(vl, ws) == 0
    _compare(eager, [o, lse, stats, lists["mask"], g])
