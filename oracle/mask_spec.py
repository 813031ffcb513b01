"""Canonical BackLite tile-selection rule (mask_from_stats), written plainly.

TEST INFRASTRUCTURE ONLY (see ``oracle/attention.py``).  Shares no code with
the CUDA path; the CUDA kernel implements the same written rule separately.

Sources: "BackLite" README, How It Works (Phase 2): for each tile pair
p_tile = exp(LSE_tile - LSE_row); the smallest-weight tiles whose cumulative
weight stays below negl_prob are skipped.  "Introducing BackLite", Using
Sparsity: neglect the smallest-weight tiles that sum to a small fraction of
the attention weight; a skipped tile costs no loads and no FLOPs.  README,
Key properties: cumulative weight < negl_prob (strict); negl_prob = 0 is the
plain dense backward.

The pages fix neither the reduction over a tile's rows, the scope of the
selection, the tie-break nor the arithmetic.  Readings adopted:

1. Per query tile i and key tile j of one (batch, query head):
   d_ij = max over rows r < n of tile i of fp32(LSE_{r,j} - LSE_r), clamped
   to <= 0 (an fp32 value; -0 becomes +0).  w_ij = exp(d_ij) is the largest
   weight any row of the tile puts on key tile j, so a row's skipped mass is
   at most the sum of the skipped w_ij.
2. w is turned into a 40-bit fixed-point integer E_ij = ceil(e_ij * 2^40)
   with e_ij = detexp(d_ij), an exp evaluated by fp32 operations that each
   round to nearest (no fused multiply-add):
     d = -inf          -> E = 0
     t = d * LOG2E_F   (fp32); if t < -48 -> E = 1 (positive, below 2^-48)
     k = rint(t) (ties to even); f = t - k (exact)
     p = Horner over the Taylor series of 2^f = sum_m (ln 2)^m f^m / m!,
         m = 0..7, coefficients C_m = fp32(round-nearest((ln 2)^m / m!))
     e = p * 2^k (exact)
3. The threshold is the integer T = ceil(negl_prob * 2^40).
4. Per query tile the non-NaN key tiles are ordered by (d ascending, j
   ascending).  The skipped set is the longest prefix of that order whose
   running integer sum of E stays < T; everything else is active.  A NaN d
   keeps its tile active and is counted.
5. With a causal or sliding-window structure, a tile none of whose (query,
   key) pairs attends is never kept, whatever negl_prob (it has nothing to
   compute; its weight is 0, so with negl_prob > 0 the rule above already
   skips it).
6. Outputs per (b, h): mask [T_r, T_c] uint8 (1 = compute), kv_idx
   [T_r, T_c] int32 (active key tiles ascending, then -1), kv_cnt [T_r],
   q_idx [T_c, T_r] int32 (active query tiles ascending, then -1), q_cnt [T_c].

Integer sums are exact, so the rule gives one answer however a parallel
implementation orders its additions.
"""
from __future__ import annotations

import math
from decimal import Decimal, getcontext

import numpy as np

FIXED_BITS = 40
TINY_T = np.float32(-48.0)


def _round_to_f32(x: Decimal) -> np.float32:
    """Round a high-precision Decimal to the nearest fp32."""
    f = np.float32(float(x))
    best, best_err = f, abs(Decimal(float(f)) - x)
    for cand in (np.nextafter(f, np.float32(np.inf)),
                 np.nextafter(f, np.float32(-np.inf))):
        err = abs(Decimal(float(cand)) - x)
        if err < best_err:
            best, best_err = cand, err
    return np.float32(best)


def _constants():
    getcontext().prec = 60
    ln2 = Decimal(2).ln()
    log2e = _round_to_f32(1 / ln2)
    coeffs = [_round_to_f32(ln2 ** m / math.factorial(m)) for m in range(8)]
    return log2e, coeffs


LOG2E_F, TAYLOR_C = _constants()


def threshold(negl_prob: float) -> int:
    """T = ceil(negl_prob * 2^40) (exact in fp64)."""
    return int(math.ceil(float(negl_prob) * float(2 ** FIXED_BITS)))


def detexp_fixed(d) -> np.ndarray:
    """E = ceil(detexp(d) * 2^40) as uint64, for fp32 d <= 0 (or -inf)."""
    d = np.asarray(d, dtype=np.float32)
    E = np.zeros(d.shape, dtype=np.uint64)
    t = d * LOG2E_F
    finite = np.isfinite(d)
    tiny = finite & (t < TINY_T)
    E[tiny] = 1
    norm = finite & ~tiny
    if np.any(norm):
        tn = t[norm]
        k = np.rint(tn)
        f = tn - k
        p = TAYLOR_C[7]
        for m in range(6, -1, -1):
            p = (p * f) + TAYLOR_C[m]
        e = np.ldexp(p.astype(np.float32), k.astype(np.int32)).astype(np.float32)
        E[norm] = np.ceil(e * np.float32(2.0 ** FIXED_BITS)).astype(np.uint64)
    return E


def tile_weights(stats_h, lse_h, n, block_q):
    """d_ij (fp32) for one (b, h): stats_h [T_c, n_pad] fp32, lse_h [n] fp32.

    Returns d [T_r, T_c] (clamped to <= 0, NaN kept) for rows r < n.
    """
    stats_h = np.asarray(stats_h, dtype=np.float32)
    lse_h = np.asarray(lse_h, dtype=np.float32)
    T_c = stats_h.shape[0]
    T_r = -(-n // block_q)
    d = np.empty((T_r, T_c), dtype=np.float32)
    for i in range(T_r):
        r0, r1 = i * block_q, min(n, (i + 1) * block_q)
        diff = stats_h[:, r0:r1] - lse_h[None, r0:r1]       # fp32, rounded
        d[i] = diff.max(axis=1)
    with np.errstate(invalid="ignore"):
        d = np.where(d > 0, np.float32(0), d)
    d = np.where(d == 0, np.float32(0), d)                  # -0 -> +0
    return d.astype(np.float32)


def select_row(d_row: np.ndarray, T: int):
    """Active flags (uint8) of one query tile's key tiles, and its NaN count."""
    T_c = d_row.shape[0]
    nan = np.isnan(d_row)
    active = np.ones(T_c, dtype=np.uint8)
    idx = np.nonzero(~nan)[0]
    if len(idx) and T > 0:
        order = idx[np.lexsort((idx, d_row[idx]))]        # d asc, then j asc
        run = np.cumsum(detexp_fixed(d_row[order]), dtype=np.uint64)
        n_skip = int(np.count_nonzero(run < np.uint64(T)))
        active[order[:n_skip]] = 0
    return active, int(nan.sum())


def structurally_empty(T_r, T_c, n, block_q, block_k, causal=False, window=0):
    """[T_r, T_c] bool: tiles in which no (query, key) pair attends."""
    empty = np.zeros((T_r, T_c), dtype=bool)
    if not (causal or window):
        return empty
    for i in range(T_r):
        r0, r1 = i * block_q, min(n, (i + 1) * block_q) - 1
        for j in range(T_c):
            c0, c1 = j * block_k, min(n, (j + 1) * block_k) - 1
            # some pair attends iff the lowest key is <= the highest row (causal)
            # and the highest key is > the lowest row - window (window)
            some = True
            if causal:
                some &= c0 <= r1
            if window:
                some &= c1 > r0 - window
            empty[i, j] = not some
    return empty


def mask_from_stats(stats, lse, n, block_q, block_k, negl_prob, causal=False, window=0):
    """Apply the rule to fp32 stats [B,H,T_c,n_pad] and fp32 LSE [B,H,n].

    Returns a dict of numpy arrays: mask, kv_idx, kv_cnt, q_idx, q_cnt, and the
    number of NaN tile weights seen.
    """
    stats = np.asarray(stats, dtype=np.float32)
    lse = np.asarray(lse, dtype=np.float32)
    B, H, T_c, _ = stats.shape
    T_r = -(-n // block_q)
    T = threshold(negl_prob)
    mask = np.ones((B, H, T_r, T_c), dtype=np.uint8)
    nan_total = 0
    empty = structurally_empty(T_r, T_c, n, block_q, block_k, causal, window)
    for b in range(B):
        for h in range(H):
            d = tile_weights(stats[b, h], lse[b, h], n, block_q)
            for i in range(T_r):
                mask[b, h, i], c = select_row(d[i], T)
                nan_total += c
            mask[b, h][empty] = 0
    return lists_from_mask(mask) | {"nan_count": nan_total}


def lists_from_mask(mask):
    """Compact a [B,H,T_r,T_c] mask into ascending per-row/per-column lists."""
    mask = np.asarray(mask, dtype=np.uint8)
    B, H, T_r, T_c = mask.shape
    kv_idx = np.full((B, H, T_r, T_c), -1, dtype=np.int32)
    q_idx = np.full((B, H, T_c, T_r), -1, dtype=np.int32)
    kv_cnt = mask.sum(axis=3, dtype=np.int32)
    q_cnt = mask.sum(axis=2, dtype=np.int32)
    for b in range(B):
        for h in range(H):
            for i in range(T_r):
                a = np.nonzero(mask[b, h, i])[0]
                kv_idx[b, h, i, :len(a)] = a
            for j in range(T_c):
                a = np.nonzero(mask[b, h, :, j])[0]
                q_idx[b, h, j, :len(a)] = a
    return {"mask": mask, "kv_idx": kv_idx, "kv_cnt": kv_cnt,
            "q_idx": q_idx, "q_cnt": q_cnt}
