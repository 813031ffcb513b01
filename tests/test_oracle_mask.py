"""Pins for the oracle's tile-selection rule (CPU only).

* detexp against math.exp, and its exact points (d = 0, d = -inf);
* hand-worked masks from the README's rule (tests/golden/mask_hand_worked.json);
* a brute-force enumeration over every subset on tiny rows: the skipped set
  must be the largest subset that is closed downward in (d, j) order and whose
  fixed-point weight stays below the threshold;
* the uniform-attention special case through the whole chain;
* per-row skipped mass < negl_prob on a clustered workload;
* negl_prob = 0 keeps everything; negl_prob -> 1 keeps a minimal suffix.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import attention as A
from oracle import mask_spec as M

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TWO40 = 2.0 ** 40


def test_detexp_tracks_exp():
    d = -np.linspace(0, 33, 20001).astype(np.float32)
    E = M.detexp_fixed(d).astype(np.float64) / TWO40
    ref = np.exp(d.astype(np.float64))
    # t = d*log2(e) is rounded to fp32, so the relative error grows like
    # |t| * 2^-24 * ln 2; the fixed-point ceiling adds at most 2^-40.
    ad = np.abs(d.astype(np.float64))
    assert np.all(np.abs(E - ref) <= (2e-7 + 6e-8 * ad) * ref + 1.0 / TWO40)
    assert np.all(E >= ref * (1 - 2e-7 - 6e-8 * ad))
    assert M.detexp_fixed(np.float32(0.0)) == 2 ** 40
    assert M.detexp_fixed(np.float32(-np.inf)) == 0
    assert M.detexp_fixed(np.float32(-50.0)) == 1         # tiny but positive
    assert np.all(np.diff(M.detexp_fixed(d).astype(np.int64)) <= 0)   # monotone


def test_threshold_is_exact_ceiling():
    assert M.threshold(0.0) == 0
    assert M.threshold(0.5) == 2 ** 39
    assert M.threshold(0.05) == math.ceil(0.05 * 2 ** 40)


def _row_stats(lse_tile):
    """One query row, LSE_row = 0: stats [T_c, 1] and lse [1]."""
    st = np.asarray(lse_tile, dtype=np.float32)[:, None]
    return st, np.zeros(1, dtype=np.float32)


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "mask_hand_worked.json")))["cases"])
def test_hand_worked_masks(case):
    if "w" in case:
        with np.errstate(divide="ignore"):
            lt = np.log(np.asarray(case["w"], dtype=np.float64))
        negl = case["negl_prob"]
    else:
        lt = case["lse_tile"]
        negl = case["negl_prob_times_2p40"] / TWO40
    st, lse = _row_stats(lt)
    out = M.mask_from_stats(st[None, None], lse[None, None], 1, 1, 1, negl)
    assert out["mask"][0, 0, 0].tolist() == case["mask"], case["why"]


def _brute_force_skip(d, T):
    """Largest subset closed downward in (d, j) order with sum(E) < T."""
    T_c = len(d)
    E = M.detexp_fixed(d).astype(object)
    best = set()
    for size in range(T_c + 1):
        for sub in itertools.combinations(range(T_c), size):
            s = set(sub)
            closed = all((d[a], a) <= (d[b], b) or b in s
                         for a in s for b in range(T_c))
            if not closed:
                continue
            if sum(E[a] for a in s) < T and len(s) >= len(best):
                best = s
    return best


@pytest.mark.parametrize("seed", range(12))
def test_selection_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    T_c = int(rng.integers(1, 8))
    w = rng.dirichlet(np.full(T_c, 0.5))
    # a few exact ties and an empty tile
    if T_c > 2:
        w[1] = w[0]
    with np.errstate(divide="ignore"):
        lt = np.log(w)
    if T_c > 3 and seed % 2:
        lt[3] = -np.inf
    negl = float(rng.choice([0.0, 0.01, 0.05, 0.2, 0.5, 0.9]))
    st, lse = _row_stats(lt)
    d = M.tile_weights(st, lse, 1, 1)[0]
    mask = M.mask_from_stats(st[None, None], lse[None, None], 1, 1, 1, negl)["mask"][0, 0, 0]
    skipped = {j for j in range(T_c) if mask[j] == 0}
    assert skipped == _brute_force_skip(list(d), M.threshold(negl))


@pytest.mark.parametrize("n,bk,negl", [(2048, 64, 0.05), (2048, 64, 0.1), (4096, 128, 0.05), (1024, 64, 0.3)])
def test_uniform_attention_skips_lowest_indices(n, bk, negl):
    """Q = 0: every key tile weighs B_c/n, so ceil(negl*T_c) - 1 tiles go, lowest j first."""
    d = 8
    q = np.zeros((1, n, 1, d))
    k = np.random.default_rng(0).standard_normal((1, n, 1, d))
    _, L, st = A.forward(q, k, k, 0.3, block_q=bk, block_k=bk)
    T_c = n // bk
    assert abs(negl * T_c - round(negl * T_c)) > 0.05        # away from the cut
    out = M.mask_from_stats(st.astype(np.float32), L.astype(np.float32), n, bk, bk, negl)
    k_skip = math.ceil(negl * T_c) - 1
    expect = np.ones(T_c, dtype=np.uint8)
    expect[:k_skip] = 0
    for i in range(n // bk):
        assert out["mask"][0, 0, i].tolist() == expect.tolist()
    assert np.all(out["kv_cnt"] == T_c - k_skip)


def _clustered(n=1024, H=2, Hk=1, d=16, seed=0):
    rng = np.random.default_rng(seed)
    mu = rng.standard_normal((16, d))
    c = (np.arange(n) // 32) % 16
    q = 2.5 * mu[c][None, :, None, :] + rng.standard_normal((1, n, H, d))
    k = 2.5 * mu[c][None, :, None, :] + rng.standard_normal((1, n, Hk, d))
    v = rng.standard_normal((1, n, Hk, d))
    return q, k, v


@pytest.mark.parametrize("negl", [0.01, 0.05, 0.1])
def test_skipped_mass_per_row_below_negl(negl):
    n, b = 1000, 64                          # ragged last tile (40 rows / keys)
    q, k, v = _clustered(n=n)
    _, L, st = A.forward(q, k, v, 0.25, block_q=b, block_k=b)
    out = M.mask_from_stats(st.astype(np.float32), L.astype(np.float32), n, b, b, negl)
    assert out["mask"].min() == 0            # the case really skips tiles
    for h in range(2):
        w = np.exp(st[0, h, :, :n] - L[0, h][None, :])     # [T_c, n]
        for r in range(n):
            skipped = out["mask"][0, h, r // b] == 0
            mass = w[skipped, r].sum()
            # fp32 rounding of the stats bounds the excess at a few 1e-6 relative
            assert mass < negl * (1 + 1e-5), (h, r, mass)


def test_negl_zero_keeps_all_and_near_one_keeps_minimal_suffix():
    n, b = 512, 64
    q, k, v = _clustered(n=n, H=1)
    _, L, st = A.forward(q, k, v, 0.25, block_q=b, block_k=b)
    st32, L32 = st.astype(np.float32), L.astype(np.float32)
    out0 = M.mask_from_stats(st32, L32, n, b, b, 0.0)
    assert np.all(out0["mask"] == 1) and np.all(out0["kv_cnt"] == n // b)
    out1 = M.mask_from_stats(st32, L32, n, b, b, 0.999)
    d = M.tile_weights(st32[0, 0], L32[0, 0], n, b)
    for i in range(n // b):
        E = M.detexp_fixed(d[i]).astype(np.float64) / TWO40
        act = out1["mask"][0, 0, i] == 1
        # the kept tiles are the heaviest ones and removing the lightest kept
        # tile would push the skipped weight to >= negl_prob
        assert E[act].min() >= E[~act].max() if (~act).any() else True
        assert E[~act].sum() + E[act].min() >= 0.999 - 1e-9


def test_nan_weight_keeps_tile_active():
    st, lse = _row_stats([np.nan, -20.0, 0.0])
    out = M.mask_from_stats(st[None, None], lse[None, None], 1, 1, 1, 0.5)
    assert out["mask"][0, 0, 0].tolist() == [1, 0, 1]
    assert out["nan_count"] == 1


def test_lists_are_ascending_compactions():
    rng = np.random.default_rng(2)
    m = (rng.random((2, 3, 5, 7)) < 0.6).astype(np.uint8)
    L = M.lists_from_mask(m)
    for b in range(2):
        for h in range(3):
            for i in range(5):
                c = L["kv_cnt"][b, h, i]
                assert list(L["kv_idx"][b, h, i, :c]) == [j for j in range(7) if m[b, h, i, j]]
                assert np.all(L["kv_idx"][b, h, i, c:] == -1)
            for j in range(7):
                c = L["q_cnt"][b, h, j]
                assert list(L["q_idx"][b, h, j, :c]) == [i for i in range(5) if m[b, h, i, j]]
                assert np.all(L["q_idx"][b, h, j, c:] == -1)


def test_structurally_empty_tiles_brute_force():
    """A tile is empty iff no (row, key) pair in it attends (checked pair by pair)."""
    n, bq, bk = 50, 8, 16
    for causal, window in ((True, 0), (True, 9), (True, 40)):
        e = M.structurally_empty(-(-n // bq), -(-n // bk), n, bq, bk, causal, window)
        for i in range(e.shape[0]):
            for j in range(e.shape[1]):
                rows = range(i * bq, min(n, (i + 1) * bq))
                cols = range(j * bk, min(n, (j + 1) * bk))
                some = any(c <= r and (window == 0 or c > r - window) for r in rows for c in cols)
                assert e[i, j] == (not some), (causal, window, i, j)


def test_causal_mask_keeps_nonempty_and_drops_empty_even_at_negl_zero():
    n, b = 512, 64
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, n, 1, 16)) * 2
    k = rng.standard_normal((1, n, 1, 16)) * 2
    _, L, st = A.forward(q, k, k, 0.25, block_q=b, block_k=b, causal=True, window=150)
    out = M.mask_from_stats(st.astype(np.float32), L.astype(np.float32), n, b, b, 0.0,
                            causal=True, window=150)
    empty = M.structurally_empty(n // b, n // b, n, b, b, True, 150)
    assert np.all(out["mask"][0, 0][empty] == 0) and np.all(out["mask"][0, 0][~empty] == 1)
