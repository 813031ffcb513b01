"""Helpers shared by the GPU parity tests: run the CUDA chain through the C
ABI binding, run the oracle on the same seeded inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

from oracle import attention as A
from oracle import mask_spec as M

# Tolerances of the parity bar: relative L2 for O and the gradients, absolute
# for the natural-log LSE.
REL_L2 = 1e-2
LSE_ABS = 1e-3
# Tile statistics: compared where the tile carries weight >= e^-STATS_WINDOW of
# its row (smaller tiles may legitimately underflow to -inf in fp32).
STATS_WINDOW = 20.0
STATS_ABS = 2e-3


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def gpu_forward(shape, q, k, v, scale, with_stats=True):
    from block_sparse_attention_fwd_gb300 import _lib
    dev = torch.device("cuda")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    B, n, H, d = q.shape
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, n), dtype=torch.float32, device=dev)
    stats = None
    if with_stats:
        stats = torch.empty(_lib.tile_stats_elems(shape), dtype=torch.float32, device=dev)
        T_r, T_c = _lib.tiles(shape)
        stats = stats.view(B, H, T_c, T_r * shape.block_q)
    _lib.attn_fwd(shape, qd, kd, vd, scale, o, lse, stats)
    return qd, kd, vd, o, lse, stats


def gpu_mask(shape, stats, lse, negl):
    from block_sparse_attention_fwd_gb300 import _lib
    lists = _lib.alloc_lists(shape, stats.device)
    _lib.mask_from_stats(shape, stats, lse, negl, lists)
    return lists


def lists_to_device(lists_np, dev="cuda"):
    out = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev)
           for k, v in lists_np.items() if k != "nan_count"}
    out["nan_count"] = torch.zeros(1, dtype=torch.int32, device=dev)
    return out


def gpu_backward(shape, qd, kd, vd, o, g_o, lse, scale, lists):
    from block_sparse_attention_fwd_gb300 import _lib
    dev = qd.device
    god = g_o.to(dev)
    g_q, g_k, g_v = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty(_lib.bwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)
    _lib.attn_bwd(shape, qd, kd, vd, o, god, lse, scale, lists, g_q, g_k, g_v, ws)
    status = _lib.bwd_check_status(shape, ws)
    return g_q, g_k, g_v, status


def cpu(t):
    return t.detach().to("cpu").float().numpy() if t.dtype == torch.bfloat16 else \
        t.detach().to("cpu").numpy()


def oracle_forward(q, k, v, scale, bq, bk):
    return A.forward(q, k, v, scale, block_q=bq, block_k=bk)


def oracle_mask(stats, lse, n, bq, bk, negl):
    return M.mask_from_stats(np.asarray(stats, dtype=np.float32),
                             np.asarray(lse, dtype=np.float32), n, bq, bk, negl)


def compare_stats(gpu_stats, or_stats, or_lse, n):
    """Max |dLSE_tile| over tiles with weight >= e^-STATS_WINDOW; and that the
    remaining ones stay small on the GPU too.  Returns (max_err, n_checked)."""
    g = np.asarray(gpu_stats, dtype=np.float64)[..., :n]
    o = np.asarray(or_stats, dtype=np.float64)[..., :n]
    L = np.asarray(or_lse, dtype=np.float64)[:, :, None, :]
    big = o > L - STATS_WINDOW
    err = np.abs(g[big] - o[big]).max() if big.any() else 0.0
    thr = np.broadcast_to(L - STATS_WINDOW + 1.0, g.shape)
    small_ok = bool(np.all(g[~big] < thr[~big]))
    return float(err), int(big.sum()), bool(small_ok)


def assert_lists_equal(gpu_lists, ref):
    for key in ("mask", "kv_idx", "kv_cnt", "q_idx", "q_cnt"):
        a = cpu(gpu_lists[key])
        b = np.asarray(ref[key])
        assert a.shape == b.shape, key
        bad = np.argwhere(a != b)
        assert len(bad) == 0, f"{key}: {len(bad)} mismatches, first at {bad[:3].tolist()}"


def to_device_like(x_np, like):
    """An oracle array as a device tensor with the dtype/shape of ``like``."""
    return torch.from_numpy(np.ascontiguousarray(x_np)).to(dtype=like.dtype,
                                                            device=like.device)
