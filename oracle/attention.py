"""Plain fp64 CPU oracle for exact attention, per-tile LSE statistics and the
masked (BackLite) attention backward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  It shares no
code with the CUDA path: no kernels, headers, helpers or constants.

Everything is written as the dense matrix definitions, one (batch, head) at a
time, with numpy matmuls as the only library step.  Query rows may be handled
in groups purely to bound memory; every group applies the same per-row
formula, so grouping changes nothing but the order of fp64 additions in the
sums over rows (G_K, G_V).

Sources (page title, section):

* "Introducing BackLite", Backpropagation for attention: the forward
  S = Q K^T / sqrt(d), P = softmax_row(S), O = P V and the backward
  G_V = P^T G_O, G_P = G_O V^T, D = diag(G_O O^T), G_S = G_P (.) P - diag(D) P,
  G_Q = G_S K / sqrt(d), G_K = G_S^T Q / sqrt(d).  A general softmax scale s
  replaces 1/sqrt(d) ("BackLite" README, Forward signature: ``scale``).
* "Introducing BackLite", Using Sparsity: the forward is exact; in the
  backward the recorded negligible entries of P are masked out, and the same
  mask serves G_V, G_S and the products with Q and K.
* "BackLite" README, How It Works: per-tile LSE for every (query, key tile)
  and p_tile = exp(LSE_tile - LSE_row).
* "Flash Attention" explainer (infinite-joy), Safe Softmax Algorithm: the
  row maximum is subtracted before exponentiating; Flash Attention Backward
  Pass: D_i = rowsum(dO_i (.) O_i), dQ = dS K, dK = dS^T Q.

Readings where the pages are silent: the LSE is the natural-log
log-sum-exp of the scaled scores s*q.k (the README's p_tile formula uses exp);
a tile LSE is taken per query row and key tile; a tile whose exponentials all
underflow has LSE -inf; rows r >= n of the last query tile do not exist and
their stats entries are -inf; D is formed from the forward output as it is
stored (bf16, see ``as_stored_output``) and P from the full-row LSE (no
renormalisation over the kept tiles).
"""
from __future__ import annotations

import numpy as np
import torch

ROW_GROUP = 2048


def _f64(x):
    """bf16/fp32 torch tensor or numpy array -> fp64 numpy (exact widening)."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def kv_head(h: int, H: int, Hk: int) -> int:
    """Key/value head that query head h reads (grouped-query attention)."""
    return h // (H // Hk)


def allowed(rows, cols, causal=False, window=0) -> np.ndarray:
    """Structural mask of the (query row, key) pairs that attend: causal keeps
    keys c <= r; a sliding window of W (with causal) keeps r - W < c <= r.
    Reading adopted for the sliding-window attention the BackLite blog trains
    with (Nanochat: windows of 1024 and 2048): W counts the query's own key."""
    r = np.asarray(rows)[:, None]
    c = np.asarray(cols)[None, :]
    ok = np.ones((r.shape[0], c.shape[1]), dtype=bool)
    if causal:
        ok &= c <= r
    if window:
        ok &= c > r - window
    return ok


def scores(q_rows: np.ndarray, k_head: np.ndarray, scale: float, rows=None, cols=None,
           causal=False, window=0) -> np.ndarray:
    """S = s * Q K^T for the given query rows against the given keys: [r, c];
    pairs the structural mask removes are -inf."""
    S = scale * (q_rows @ k_head.T)
    if causal or window:
        S = np.where(allowed(rows, cols, causal, window), S, -np.inf)
    return S


def row_softmax_stats(S: np.ndarray):
    """Safe softmax pieces of each row: max m, P = exp(S - m)/l, LSE = m + log l."""
    m = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)
    l = E.sum(axis=1, keepdims=True)
    return m[:, 0], E / l, (m + np.log(l))[:, 0]


def tile_lse(S: np.ndarray, block_k: int) -> np.ndarray:
    """Per (row, key tile) LSE: LSE_{r,j} = log sum_{c in tile j} exp(S_rc).

    Returned as [T_c, r] (key-tile major).  Computed relative to the row max
    m_r; a tile whose terms all underflow gives log 0 = -inf.
    """
    r, n = S.shape
    T_c = -(-n // block_k)
    m = S.max(axis=1, keepdims=True)
    E = np.zeros((r, T_c * block_k))
    E[:, :n] = np.exp(S - m)
    sums = E.reshape(r, T_c, block_k).sum(axis=2)          # [r, T_c]
    with np.errstate(divide="ignore"):
        out = m + np.log(sums)
    return out.T.copy()


def forward_head(q_h, k_h, v_h, scale, rows=None, block_k=None, causal=False, window=0):
    """Exact attention for one (batch, head).

    q_h [n, d], k_h/v_h [n, d] fp64.  ``rows``: query row indices (default all).
    Returns O [r, d], LSE [r] and, when ``block_k`` is given, tile stats [T_c, r].
    """
    n = q_h.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows)
    outs_o, outs_l, outs_t = [], [], []
    for g in range(0, len(rows), ROW_GROUP):
        rr = rows[g:g + ROW_GROUP]
        S = scores(q_h[rr], k_h, scale, rr, np.arange(n), causal, window)
        _, P, lse = row_softmax_stats(S)
        outs_o.append(P @ v_h)
        outs_l.append(lse)
        if block_k is not None:
            outs_t.append(tile_lse(S, block_k))
    O = np.concatenate(outs_o, axis=0)
    L = np.concatenate(outs_l, axis=0)
    T = np.concatenate(outs_t, axis=1) if block_k is not None else None
    return O, L, T


def forward(q, k, v, scale, block_q=None, block_k=None, causal=False, window=0):
    """Exact attention over BSHD tensors.

    q [B,n,H,d], k/v [B,n,Hk,d] -> O [B,n,H,d] fp64, LSE [B,H,n] fp64 and, when
    tile sizes are given, tile stats [B,H,T_c,T_r*block_q] (rows >= n are -inf).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, n, H, d = q.shape
    Hk = k.shape[2]
    O = np.zeros((B, n, H, d))
    LSE = np.zeros((B, H, n))
    stats = None
    if block_k is not None:
        T_r, T_c = -(-n // block_q), -(-n // block_k)
        stats = np.full((B, H, T_c, T_r * block_q), -np.inf)
    for b in range(B):
        for h in range(H):
            hk = kv_head(h, H, Hk)
            o, l, t = forward_head(q[b, :, h], k[b, :, hk], v[b, :, hk], scale,
                                   block_k=block_k, causal=causal, window=window)
            O[b, :, h] = o
            LSE[b, h] = l
            if stats is not None:
                stats[b, h, :, :n] = t
    return O, LSE, stats


def as_stored_output(O) -> np.ndarray:
    """The forward output as the method hands it on: the output tensor has the
    inputs' dtype (bf16), so O is the exact result rounded to nearest-even
    bf16.  D = rowsum(G_O (.) O) in the backward is formed from this stored O,
    the same tensor any caller passes back in."""
    t = torch.from_numpy(np.ascontiguousarray(O, dtype=np.float64)).to(torch.bfloat16)
    return t.double().numpy()


def element_mask(tile_mask: np.ndarray, block_q: int, block_k: int,
                 rows: np.ndarray, cols: np.ndarray) -> np.ndarray:
    """Expand a [T_r, T_c] tile mask to the element mask M[rows][:, cols]."""
    return tile_mask[np.asarray(rows)[:, None] // block_q,
                     np.asarray(cols)[None, :] // block_k].astype(np.float64)


def backward_head(q_h, k_h, v_h, o_h, go_h, lse_h, scale, tile_mask,
                  block_q, block_k, rows=None, cols=None, causal=False, window=0):
    """Masked attention backward for one (batch, query head).

    With P the exact softmax (recomputed from the full-row LSE) and M the
    element mask expanded from ``tile_mask`` (None = keep every tile):

        P^ = P (.) M,  D_r = sum_d G_O[r,d] O[r,d],  G_V = P^T G_O,
        G_P = G_O V^T, G_S = P^ (.) (G_P - D 1^T),
        G_Q = s G_S K, G_K = s G_S^T Q.

    ``rows``/``cols`` restrict the query rows and key columns that are
    formed.  G_Q [len(rows), d] is complete only when ``cols`` is every key;
    G_K, G_V [len(cols), d] are complete only when ``rows`` is every query.
    """
    n = q_h.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows)
    cols = np.arange(n) if cols is None else np.asarray(cols)
    d = q_h.shape[1]
    gq = np.zeros((len(rows), d))
    gk = np.zeros((len(cols), d))
    gv = np.zeros((len(cols), d))
    k_c, v_c = k_h[cols], v_h[cols]
    for g in range(0, len(rows), ROW_GROUP):
        rr = rows[g:g + ROW_GROUP]
        S = scores(q_h[rr], k_c, scale, rr, cols, causal, window)
        P = np.exp(S - lse_h[rr][:, None])
        if tile_mask is not None:
            P = P * element_mask(tile_mask, block_q, block_k, rr, cols)
        Dr = np.sum(go_h[rr] * o_h[rr], axis=1)
        GP = go_h[rr] @ v_c.T
        GS = P * (GP - Dr[:, None])
        gv += P.T @ go_h[rr]
        gk += scale * (GS.T @ q_h[rr])
        gq[g:g + len(rr)] = scale * (GS @ k_c)
    return gq, gk, gv


def backward(q, k, v, o, g_o, lse, scale, tile_masks=None, block_q=None,
             block_k=None, causal=False, window=0):
    """Masked attention backward over BSHD tensors (full, every row/column).

    ``tile_masks``: [B, H, T_r, T_c] (nonzero = compute), or None for dense.
    ``o`` is the forward output as stored (``as_stored_output`` of the oracle's
    own O) and ``lse`` the oracle's own LSE.  Returns fp64
    G_Q [B,n,H,d], G_K and G_V [B,n,Hk,d]; the gradient of a kv head sums the
    contributions of every query head in its group.
    """
    q, k, v, o, g_o = (_f64(x) for x in (q, k, v, o, g_o))
    lse = _f64(lse)
    B, n, H, d = q.shape
    Hk = k.shape[2]
    gq = np.zeros_like(q)
    gk = np.zeros_like(k)
    gv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            hk = kv_head(h, H, Hk)
            tm = None if tile_masks is None else np.asarray(tile_masks[b, h])
            a, bk, bv = backward_head(q[b, :, h], k[b, :, hk], v[b, :, hk],
                                      o[b, :, h], g_o[b, :, h], lse[b, h], scale,
                                      tm, block_q, block_k, causal=causal, window=window)
            gq[b, :, h] = a
            gk[b, :, hk] += bk
            gv[b, :, hk] += bv
    return gq, gk, gv


def combine(o_parts, lse_parts):
    """Merge partial attention results over disjoint key sets ("BackLite"
    README, Key properties: the LSE output serves to combine partial results).

    o_parts [P, B, n, H, d], lse_parts [P, B, H, n] (natural log) ->
    O = sum_p exp(LSE_p - LSE) O_p with LSE = log sum_p exp(LSE_p).
    Parts with LSE -inf carry no weight; rows where every part is -inf get
    O = 0 and LSE = -inf.
    """
    o_parts = _f64(o_parts)
    lse_parts = _f64(lse_parts)
    m = lse_parts.max(axis=0)                               # [B, H, n]
    finite = np.isfinite(m)
    mm = np.where(finite, m, 0.0)
    with np.errstate(invalid="ignore"):
        w = np.exp(lse_parts - mm[None])                    # [P, B, H, n]
    w = np.where(np.isfinite(lse_parts), w, 0.0)
    tot = w.sum(axis=0)
    lse = np.where(finite, mm + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    wn = np.where(tot[None] > 0, w / np.where(tot > 0, tot, 1.0)[None], 0.0)
    # weights are per (b, h, row); outputs are (b, row, h, d)
    o = np.einsum("pbhn,pbnhd->bnhd", wn, o_parts)
    return o, lse


def forward_keys(q, k, v, scale, keys):
    """Exact attention of every query over the key subset `keys` only:
    O [B,n,H,d] and LSE [B,H,n] (-inf where the subset is empty)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, n, H, d = q.shape
    Hk = k.shape[2]
    keys = np.asarray(keys)
    O = np.zeros((B, n, H, d))
    L = np.full((B, H, n), -np.inf)
    if len(keys) == 0:
        return O, L
    for b in range(B):
        for h in range(H):
            hk = kv_head(h, H, Hk)
            S = scores(q[b, :, h], k[b, keys, hk], scale)
            _, P, lse = row_softmax_stats(S)
            O[b, :, h] = P @ v[b, keys, hk]
            L[b, h] = lse
    return O, L
