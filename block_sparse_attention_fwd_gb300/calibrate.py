"""Choose negl_prob for a workload from the gradients it produces.

"Introducing BackLite" (Using Sparsity; Experiments) judges the sparse
backward by the cosine similarity and the relative L2 error of its gradients
against the dense backward, reports more than 50% of the tiles skipped at
cos > 0.99 and rel-L2 < 0.1 on a video model, and proposes tuning negl_prob
to such a target as training goes.  ``calibrate_negl_prob`` does that for one
batch: it runs the forward with tile statistics and the dense backward once,
then mask + sparse backward for every candidate negl_prob, measures the three
gradients against the dense ones (``bl_grad_error``), and returns the largest
candidate whose worst gradient meets the target.

Every step runs in libbl_attn.so; this module orders the calls and applies
the selection rule (``select_negl``), which is plain host logic.
"""
from __future__ import annotations

import dataclasses

import torch

from . import _lib


@dataclasses.dataclass
class Trial:
    negl_prob: float
    skip_frac: float          # fraction of structurally non-empty tiles skipped
    rel_l2: dict              # gradient name -> relative L2 error vs the dense backward
    cos: dict                 # gradient name -> cosine similarity vs the dense backward

    @property
    def worst_rel_l2(self) -> float:
        return max(self.rel_l2.values())

    @property
    def worst_cos(self) -> float:
        return min(self.cos.values())


def select_negl(trials, max_rel_l2: float = 0.1, min_cos: float = 0.99):
    """The largest negl_prob among ``trials`` whose worst gradient has
    rel-L2 <= max_rel_l2 and cos >= min_cos; 0.0 (the dense backward) when none
    does.  The errors need not grow monotonically with negl_prob, so every
    trial is checked rather than stopping at the first failure."""
    ok = [t.negl_prob for t in trials if t.worst_rel_l2 <= max_rel_l2 and t.worst_cos >= min_cos]
    return max(ok) if ok else 0.0


def calibrate_negl_prob(q, k, v, g_o, *, candidates=(0.005, 0.01, 0.02, 0.05, 0.1, 0.2),
                        max_rel_l2: float = 0.1, min_cos: float = 0.99, scale=None,
                        block: int = 128, causal: bool = False, window: int = 0):
    """Returns (negl_prob, trials) for bf16 device tensors q, g_o [B,n,H,d] and
    k, v [B,n,Hk,d]."""
    B, n, H, d = q.shape
    Hk = k.shape[2]
    if scale is None:
        scale = d ** -0.5
    shape = _lib.make_shape(B, n, H, Hk, d, block, block, int(causal), int(window))
    T_r, T_c = _lib.tiles(shape)
    dev = q.device
    o = torch.empty_like(q)
    lse = torch.empty((B, H, n), dtype=torch.float32, device=dev)
    stats = torch.empty((B, H, T_c, T_r * block), dtype=torch.float32, device=dev)
    _lib.attn_fwd(shape, q, k, v, scale, o, lse, stats)
    ws = torch.empty(_lib.bwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)
    ref = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    _lib.attn_bwd(shape, q, k, v, o, g_o, lse, scale, None, *ref, ws)
    got = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    lists = _lib.alloc_lists(shape, dev)
    # tiles with at least one attending pair (all of them without causal structure)
    dense_lists = _lib.alloc_lists(shape, dev)
    _lib.mask_from_stats(shape, stats, lse, 0.0, dense_lists)
    nonempty = float(dense_lists["mask"].sum())
    out = torch.empty(4, dtype=torch.float64, device=dev)
    trials = []
    for negl in sorted(candidates):
        _lib.mask_from_stats(shape, stats, lse, float(negl), lists)
        _lib.attn_bwd(shape, q, k, v, o, g_o, lse, scale, lists, *got, ws)
        rel, cos = {}, {}
        for name, a, b in zip(("G_Q", "G_K", "G_V"), got, ref):
            rel[name], cos[name] = _lib.grad_error(a, b, out)
        kept = float(lists["mask"].sum())
        trials.append(Trial(float(negl), 1.0 - kept / nonempty if nonempty else 0.0, rel, cos))
    return select_negl(trials, max_rel_l2, min_cos), trials
