"""Pins for the oracle's exact forward and per-tile LSE statistics (CPU only).

Each check compares the oracle with something other than itself: a library
routine for the dense special case, a closed form, an invariant, or a
pure-Python brute force on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_safe_softmax_survives_page_overflow_example():
    g = json.load(open(os.path.join(GOLDEN, "softmax_overflow.json")))
    S = np.array([g["x"]])
    m, P, lse = A.row_softmax_stats(S)
    assert np.all(np.isfinite(P)) and np.isfinite(lse[0])
    ref = [math.exp(v) for v in g["shift_invariant_equivalent"]]
    ref = np.array(ref) / sum(ref)
    assert np.allclose(P[0], ref, rtol=0, atol=1e-15)
    assert abs(lse[0] - (1002.0 + math.log(sum(math.exp(v - 2.0) for v in [0.0, 1.0, 2.0])))) < 1e-12


@pytest.mark.parametrize("B,n,H,Hk,d", [(1, 7, 1, 1, 4), (2, 19, 4, 2, 8), (1, 33, 3, 1, 16)])
def test_forward_matches_torch_sdpa_fp64(B, n, H, Hk, d):
    q, k, v = _rand((B, n, H, d), 1), _rand((B, n, Hk, d), 2), _rand((B, n, Hk, d), 3)
    scale = 0.37
    O, L, _ = A.forward(q, k, v, scale)
    G = H // Hk
    qt = torch.from_numpy(q).permute(0, 2, 1, 3)
    kt = torch.from_numpy(k).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    vt = torch.from_numpy(v).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    assert np.allclose(O, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-13)
    lse_ref = torch.logsumexp(scale * qt @ kt.transpose(-1, -2), dim=-1).numpy()
    assert np.allclose(L, lse_ref, rtol=0, atol=1e-12)


def test_tile_stats_brute_force_tiny():
    n, d, bk, bq = 10, 3, 4, 4
    q, k, v = _rand((1, n, 1, d), 4), _rand((1, n, 1, d), 5), _rand((1, n, 1, d), 6)
    scale = 0.8
    _, _, st = A.forward(q, k, v, scale, block_q=bq, block_k=bk)
    T_c, T_r = 3, 3
    assert st.shape == (1, 1, T_c, T_r * bq)
    for r in range(n):
        for j in range(T_c):
            tot = 0.0
            for c in range(j * bk, min(n, (j + 1) * bk)):
                dot = sum(q[0, r, 0, x] * k[0, c, 0, x] for x in range(d))
                tot += math.exp(scale * dot)
            assert abs(st[0, 0, j, r] - math.log(tot)) < 1e-12
    assert np.all(st[0, 0, :, n:] == -np.inf)     # rows past n do not exist


def test_tile_stats_partition_invariant():
    """sum_j exp(LSE_{r,j} - LSE_r) = 1 and logsumexp_j LSE_{r,j} = LSE_r."""
    n, d = 300, 16
    q = 3 * _rand((1, n, 2, d), 7)
    k = 3 * _rand((1, n, 1, d), 8)
    v = _rand((1, n, 1, d), 9)
    _, L, st = A.forward(q, k, v, 0.25, block_q=64, block_k=64)
    for h in range(2):
        w = np.exp(st[0, h, :, :n] - L[0, h][None, :])
        assert np.max(np.abs(w.sum(axis=0) - 1.0)) < 1e-12
        m = st[0, h, :, :n].max(axis=0)
        lse2 = m + np.log(np.exp(st[0, h, :, :n] - m).sum(axis=0))
        assert np.max(np.abs(lse2 - L[0, h])) < 1e-11


@pytest.mark.parametrize("n,bk", [(256, 64), (250, 64), (129, 128)])
def test_uniform_attention_closed_form(n, bk):
    """Q = 0 gives S = 0: LSE_r = log n and LSE_{r,j} = log(#keys in tile j)."""
    d = 8
    q = np.zeros((1, n, 1, d))
    k, v = _rand((1, n, 1, d), 10), _rand((1, n, 1, d), 11)
    O, L, st = A.forward(q, k, v, 0.125, block_q=bk, block_k=bk)
    assert np.allclose(L, math.log(n), atol=1e-13)
    assert np.allclose(O[0, :, 0], v[0, :, 0].mean(axis=0)[None, :], atol=1e-13)
    T_c = -(-n // bk)
    for j in range(T_c):
        cnt = min(n, (j + 1) * bk) - j * bk
        assert np.allclose(st[0, 0, j, :n], math.log(cnt), atol=1e-13)


def test_underflowing_tile_is_minus_inf():
    """A key tile whose scores sit ~1e4 below the row max has LSE_tile = -inf."""
    n, d = 8, 1
    q = np.ones((1, n, 1, d))
    k = np.zeros((1, n, 1, d))
    k[0, :4, 0, 0] = -1.0e4
    v = np.zeros((1, n, 1, d))
    _, L, st = A.forward(q, k, v, 1.0, block_q=4, block_k=4)
    assert np.all(st[0, 0, 0, :n] == -np.inf)
    assert np.allclose(st[0, 0, 1, :n], math.log(4.0))
    assert np.allclose(L, math.log(4.0))


@pytest.mark.parametrize("cuts", [[0, 13, 40], [0, 1, 2, 40], [0, 40, 40]])
def test_combine_of_a_key_partition_is_the_full_attention(cuts):
    """Splitting the keys into disjoint sets and combining the partial results
    with their LSEs gives the full attention (and an empty part is ignored)."""
    n, d = 40, 8
    q, k, v = _rand((2, n, 4, d), 21), _rand((2, n, 2, d), 22), _rand((2, n, 2, d), 23)
    scale = 0.4
    O, L, _ = A.forward(q, k, v, scale)
    parts = [A.forward_keys(q, k, v, scale, np.arange(a, b)) for a, b in zip(cuts[:-1], cuts[1:])]
    Oc, Lc = A.combine(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    assert np.allclose(Oc, O, atol=1e-13) and np.allclose(Lc, L, atol=1e-13)


def test_combine_closed_form_and_empty_rows():
    o = np.zeros((2, 1, 1, 1, 2))
    o[0, 0, 0, 0] = [1.0, 0.0]
    o[1, 0, 0, 0] = [0.0, 1.0]
    lse = np.array([math.log(1.0), math.log(3.0)]).reshape(2, 1, 1, 1)
    Oc, Lc = A.combine(o, lse)
    assert np.allclose(Oc[0, 0, 0], [0.25, 0.75]) and abs(Lc[0, 0, 0] - math.log(4.0)) < 1e-15
    Oe, Le = A.combine(o, np.full((2, 1, 1, 1), -np.inf))
    assert np.all(Oe == 0) and Le[0, 0, 0] == -np.inf


@pytest.mark.parametrize("window", [0, 5, 17])
def test_causal_and_window_forward_match_torch(window):
    """Causal (and causal sliding-window) attention against fp64 torch SDPA with
    an explicit boolean mask; tile statistics keep their partition invariant."""
    B, n, H, Hk, d = 1, 37, 2, 1, 8
    q, k, v = _rand((B, n, H, d), 31), _rand((B, n, Hk, d), 32), _rand((B, n, Hk, d), 33)
    scale = 0.45
    O, L, st = A.forward(q, k, v, scale, block_q=8, block_k=8, causal=True, window=window)
    r = np.arange(n)[:, None]
    c = np.arange(n)[None, :]
    m = (c <= r) & ((c > r - window) if window else True)
    qt = torch.from_numpy(q).permute(0, 2, 1, 3)
    kt = torch.from_numpy(k).permute(0, 2, 1, 3).repeat_interleave(H // Hk, dim=1)
    vt = torch.from_numpy(v).permute(0, 2, 1, 3).repeat_interleave(H // Hk, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(m),
                                                           scale=scale)
    assert np.allclose(O, ref.permute(0, 2, 1, 3).numpy(), atol=1e-13)
    if window == 0:
        ref2 = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True,
                                                                scale=scale)
        assert np.allclose(O, ref2.permute(0, 2, 1, 3).numpy(), atol=1e-13)
    for h in range(H):
        w = np.exp(st[0, h, :, :n] - L[0, h][None, :])
        assert np.max(np.abs(w.sum(axis=0) - 1.0)) < 1e-12
    # a key tile wholly after the row (causal) has no weight
    assert np.all(st[0, 0, 4, :8] == -np.inf)
