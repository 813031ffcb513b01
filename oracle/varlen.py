"""Plain fp64 CPU oracle for packed variable-length batches.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  It shares no
code with the CUDA path.

The BackLite pages train on fixed-length batches and never pack sequences.
The reading taken here is the plain one: in a packed batch a query attends
only to the keys of its own sequence, so every quantity of a sequence is the
fixed-length quantity of that sequence alone (B = 1, n = its length).  The
per-sequence arrays are stored one sequence after another:

* q, k, v, o and the gradients: [total, heads, d], rows of sequence s at
  tokens cu[s] .. cu[s+1]-1;
* lse: a [H, n_s] block per sequence, at element offset H * cu[s];
* tile statistics: a [H, T_c(s), T_r(s)*block_q] block per sequence;
* mask, kv_idx: [H, T_r(s), T_c(s)]; kv_cnt: [H, T_r(s)];
  q_idx: [H, T_c(s), T_r(s)]; q_cnt: [H, T_c(s)], blocks back to back.

Each function loops over the sequences and applies the fixed-length oracle
(``attention``, ``mask_spec``) to the sequence's slice.
"""
from __future__ import annotations

import numpy as np

from . import attention as A
from . import mask_spec as M


def lengths(cu):
    cu = [int(x) for x in cu]
    return [b - a for a, b in zip(cu[:-1], cu[1:])]


def layout(cu, H, block_q, block_k):
    """Per sequence: (token offset, n, T_r, T_c) and the element offsets of its
    lse, stats, mask/kv_idx, kv_cnt, q_idx and q_cnt blocks; plus the totals."""
    cu = [int(x) for x in cu]
    offs = {"stats": 0, "mask": 0, "kv_cnt": 0, "q_idx": 0, "q_cnt": 0}
    seqs = []
    for s, n in enumerate(lengths(cu)):
        T_r, T_c = -(-n // block_q), -(-n // block_k)
        seqs.append(dict(tok=cu[s], n=n, T_r=T_r, T_c=T_c, lse=H * cu[s], **offs))
        offs["stats"] += H * T_c * T_r * block_q
        offs["mask"] += H * T_r * T_c
        offs["kv_cnt"] += H * T_r
        offs["q_idx"] += H * T_c * T_r
        offs["q_cnt"] += H * T_c
    totals = dict(offs, total=cu[-1], lse=H * cu[-1])
    return seqs, totals


def forward(q, k, v, cu, scale, block_q=None, block_k=None, causal=False, window=0):
    """Exact attention of every packed sequence: q [total,H,d], k/v
    [total,Hk,d] -> O [total,H,d], flat lse [H*total] and, when tile sizes are
    given, flat tile statistics (fp64)."""
    q, k, v = A._f64(q), A._f64(k), A._f64(v)
    total, H, d = q.shape
    seqs, tot = layout(cu, H, block_q or 1, block_k or 1)
    O = np.zeros((total, H, d))
    lse = np.zeros(tot["lse"])
    stats = np.full(tot["stats"], -np.inf) if block_k is not None else None
    for s in seqs:
        if s["n"] == 0:
            continue
        a, n = s["tok"], s["n"]
        o_s, l_s, st_s = A.forward(q[None, a:a + n], k[None, a:a + n], v[None, a:a + n], scale,
                                   block_q, block_k, causal, window)
        O[a:a + n] = o_s[0]
        lse[s["lse"]:s["lse"] + H * n] = l_s[0].reshape(-1)
        if stats is not None:
            stats[s["stats"]:s["stats"] + st_s[0].size] = st_s[0].reshape(-1)
    return O, lse, stats


def mask_from_stats(stats, lse, cu, H, block_q, block_k, negl_prob, causal=False, window=0):
    """The selection rule applied to each sequence's own fp32 statistics and
    LSE.  Returns flat arrays mask, kv_idx, kv_cnt, q_idx, q_cnt and the total
    NaN count."""
    stats = np.asarray(stats, dtype=np.float32)
    lse = np.asarray(lse, dtype=np.float32)
    seqs, tot = layout(cu, H, block_q, block_k)
    out = {"mask": np.zeros(tot["mask"], np.uint8), "kv_idx": np.zeros(tot["mask"], np.int32),
           "kv_cnt": np.zeros(tot["kv_cnt"], np.int32),
           "q_idx": np.zeros(tot["q_idx"], np.int32),
           "q_cnt": np.zeros(tot["q_cnt"], np.int32), "nan_count": 0}
    for s in seqs:
        n, T_r, T_c = s["n"], s["T_r"], s["T_c"]
        if n == 0:
            continue
        st = stats[s["stats"]:s["stats"] + H * T_c * T_r * block_q].reshape(1, H, T_c, -1)
        ls = lse[s["lse"]:s["lse"] + H * n].reshape(1, H, n)
        r = M.mask_from_stats(st, ls, n, block_q, block_k, negl_prob, causal, window)
        for key, off in (("mask", "mask"), ("kv_idx", "mask"), ("kv_cnt", "kv_cnt"),
                         ("q_idx", "q_idx"), ("q_cnt", "q_cnt")):
            flat = np.asarray(r[key]).reshape(-1)
            out[key][s[off]:s[off] + flat.size] = flat
        out["nan_count"] += r["nan_count"]
    return out


def backward(q, k, v, o, g_o, lse, cu, scale, masks=None, block_q=None, block_k=None,
             causal=False, window=0):
    """Masked attention backward of every packed sequence.  ``masks``: flat
    uint8 tile masks in the packed layout, or None for dense.  Returns G_Q
    [total,H,d], G_K and G_V [total,Hk,d] (fp64)."""
    q, k, v, o, g_o = (A._f64(x) for x in (q, k, v, o, g_o))
    lse = A._f64(lse)
    total, H, d = q.shape
    seqs, _ = layout(cu, H, block_q or 1, block_k or 1)
    gq, gk, gv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for s in seqs:
        n = s["n"]
        if n == 0:
            continue
        a = s["tok"]
        sl = slice(a, a + n)
        tm = None
        if masks is not None:
            tm = np.asarray(masks)[s["mask"]:s["mask"] + H * s["T_r"] * s["T_c"]]
            tm = tm.reshape(1, H, s["T_r"], s["T_c"])
        ls = lse[s["lse"]:s["lse"] + H * n].reshape(1, H, n)
        a_, b_, c_ = A.backward(q[None, sl], k[None, sl], v[None, sl], o[None, sl],
                                g_o[None, sl], ls, scale, tm, block_q, block_k, causal, window)
        gq[sl], gk[sl], gv[sl] = a_[0], b_[0], c_[0]
    return gq, gk, gv
