"""GPU parity of bl_lse_combine against the oracle: partial results of the
same queries over disjoint key sets (computed by the oracle, rounded to the
stored dtypes) merged on the GPU must equal the oracle's merge and, up to
the bf16 rounding of the parts, the full attention."""
import numpy as np
import pytest
import torch

from block_sparse_attention_fwd_gb300 import inputs
from oracle import attention as A
from tests import parity_util as U

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,cuts", [(128, [0, 300, 1000]), (64, [0, 1, 511, 777]),
                                    (128, [0, 1000, 1000])])
def test_combine_matches_oracle(d, cuts):
    import __graft_entry__ as g
    g.build()
    from block_sparse_attention_fwd_gb300 import _lib
    n = cuts[-1]
    w = inputs.custom("combine", B=2, n=n, H=4, Hk=2, d=d, run=40, clusters=6, alpha=3.0)
    q, k, v, _ = inputs.generate(w, seed=5, with_grad_out=False)
    parts = [A.forward_keys(q, k, v, w.scale, np.arange(a, b)) for a, b in zip(cuts[:-1], cuts[1:])]
    o_parts = np.stack([A.as_stored_output(p[0]) for p in parts])      # bf16 values
    lse_parts = np.stack([p[1] for p in parts]).astype(np.float32)
    ref_o, ref_l = A.combine(o_parts, lse_parts.astype(np.float64))
    dev = torch.device("cuda")
    op = torch.from_numpy(o_parts).to(torch.bfloat16).to(dev)
    lp = torch.from_numpy(lse_parts).to(dev)
    o = torch.empty((w.B, n, w.H, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, n), dtype=torch.float32, device=dev)
    _lib.lse_combine(op, lp, o, lse)
    assert U.rel_l2(U.cpu(o), ref_o) <= U.REL_L2
    assert np.abs(U.cpu(lse) - ref_l).max() <= U.LSE_ABS
    full_o, full_l, _ = A.forward(q, k, v, w.scale)
    assert U.rel_l2(U.cpu(o), full_o) <= U.REL_L2
    assert np.abs(U.cpu(lse) - full_l).max() <= U.LSE_ABS


def test_combine_rows_with_no_keys():
    import __graft_entry__ as g
    g.build()
    from block_sparse_attention_fwd_gb300 import _lib
    dev = torch.device("cuda")
    op = torch.randn((2, 1, 8, 1, 64), device=dev).to(torch.bfloat16)
    lp = torch.full((2, 1, 1, 8), -float("inf"), device=dev)
    lp[0, 0, 0, 3] = 0.5
    o = torch.empty((1, 8, 1, 64), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((1, 1, 8), dtype=torch.float32, device=dev)
    _lib.lse_combine(op, lp, o, lse)
    assert torch.isinf(lse[0, 0, torch.arange(8) != 3]).all()
    assert (o[0, torch.arange(8) != 3] == 0).all()
    assert torch.allclose(o[0, 3].float(), op[0, 0, 3].float()) and abs(float(lse[0, 0, 3]) - 0.5) < 1e-6
