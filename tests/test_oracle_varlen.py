"""Pins for the packed variable-length oracle (CPU only).

The oracle slices the packed tensors per sequence and calls the fixed-length
oracle.  The pins restate packing in a different form: one attention over
the whole packed token axis whose scores are masked block-diagonally (a query
sees only its own sequence's keys, at positions relative to the sequence
start), computed with torch fp64 ops and autograd.  A wrong token offset,
lse/stats/list block offset or a sequence leaking into its neighbour fails
one of them.  The layout totals are checked against a hand count.
"""
import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import mask_spec as M
from oracle import varlen as V


def _packed(cu, H, Hk, d, seed):
    rng = np.random.default_rng(seed)
    T = cu[-1]
    return (1.3 * rng.standard_normal((T, H, d)), 1.3 * rng.standard_normal((T, Hk, d)),
            rng.standard_normal((T, Hk, d)), rng.standard_normal((T, H, d)))


def _allowed(cu, causal, window):
    """[T, T] bool: query token r may attend to key token c."""
    T = cu[-1]
    seq = np.zeros(T, dtype=np.int64)
    pos = np.zeros(T, dtype=np.int64)
    for s in range(len(cu) - 1):
        seq[cu[s]:cu[s + 1]] = s
        pos[cu[s]:cu[s + 1]] = np.arange(cu[s + 1] - cu[s])
    ok = seq[:, None] == seq[None, :]
    if causal:
        ok &= pos[None, :] <= pos[:, None]
    if window:
        ok &= pos[None, :] > pos[:, None] - window
    return ok


def _block_diag_attention(q, k, v, cu, scale, causal=False, window=0):
    """torch fp64 tensors in, (O [T,H,d], LSE [H,T], S [H,T,T] masked scores)."""
    H, Hk = q.shape[1], k.shape[1]
    kk = k.repeat_interleave(H // Hk, dim=1)
    vv = v.repeat_interleave(H // Hk, dim=1)
    S = scale * torch.einsum("rhd,chd->hrc", q, kk)
    S = S.masked_fill(~torch.from_numpy(_allowed(cu, causal, window))[None], -torch.inf)
    lse = torch.logsumexp(S, dim=-1)
    O = torch.einsum("hrc,chd->rhd", torch.softmax(S, dim=-1), vv)
    return O, lse, S


CASES = [
    ([0, 5, 5, 17, 30, 30, 43], False, 0),    # empty sequences, ragged lengths, equal run
    ([0, 9, 18, 27], False, 0),                 # all equal
    ([0, 1, 21, 40], True, 0),                  # causal, length-1 sequence
    ([0, 23, 30, 52], True, 6),                 # causal sliding window
]


@pytest.mark.parametrize("cu,causal,window", CASES)
def test_forward_matches_block_diagonal_attention(cu, causal, window):
    H, Hk, d, bq, bk = 4, 2, 5, 8, 4
    q, k, v, _ = _packed(cu, H, Hk, d, seed=len(cu))
    scale = 0.6
    O, lse, stats = V.forward(q, k, v, cu, scale, bq, bk, causal, window)
    O_t, L_t, S_t = _block_diag_attention(*(torch.from_numpy(x) for x in (q, k, v)), cu, scale,
                                          causal, window)
    assert np.allclose(O, O_t.numpy(), rtol=0, atol=1e-12)
    # offsets as documented: lse block of sequence s at H * cu[s]; statistics
    # blocks [H, T_c, T_r * bq] back to back
    assert lse.size == H * cu[-1]
    st_off = 0
    for a, b in zip(cu[:-1], cu[1:]):
        n = b - a
        T_r, T_c = -(-n // bq), -(-n // bk)
        blk = lse[H * a:H * a + H * n].reshape(H, n)
        assert np.allclose(blk, L_t[:, a:a + n].numpy(), rtol=0, atol=1e-12)
        # tile statistics: log-sum-exp of the row's scores over the key tile's
        # columns, key tiles counted from the sequence start
        st = stats[st_off:st_off + H * T_c * T_r * bq].reshape(H, T_c, T_r * bq)
        st_off += H * T_c * T_r * bq
        for j in range(T_c):
            c0, c1 = a + j * bk, a + min((j + 1) * bk, n)
            want = torch.logsumexp(S_t[:, a:a + n, c0:c1], dim=-1).numpy()
            assert np.allclose(st[:, j, :n], want, rtol=0, atol=1e-12)
            assert np.all(st[:, j, n:] == -np.inf)
    assert st_off == stats.size


@pytest.mark.parametrize("cu,causal,window", CASES)
def test_backward_matches_block_diagonal_autograd(cu, causal, window):
    H, Hk, d = 4, 2, 5
    q, k, v, go = _packed(cu, H, Hk, d, seed=10 + len(cu))
    scale = 0.45
    O, lse, _ = V.forward(q, k, v, cu, scale, causal=causal, window=window)
    gq, gk, gv = V.backward(q, k, v, O, go, lse, cu, scale, causal=causal, window=window)
    tq, tk, tv = (torch.from_numpy(x).clone().requires_grad_(True) for x in (q, k, v))
    O_t, _, _ = _block_diag_attention(tq, tk, tv, cu, scale, causal, window)
    O_t.backward(torch.from_numpy(go))
    for mine, ref in ((gq, tq.grad), (gk, tk.grad), (gv, tv.grad)):
        assert np.allclose(mine, ref.numpy(), rtol=0, atol=1e-12)


def test_masked_backward_uses_each_sequences_own_tiles():
    """Tile (i, j) of sequence s covers query tokens a + i*bq.. and key tokens
    a + j*bk.. of that sequence: expand every sequence's tile mask onto the
    packed [T, T] grid and form the masked gradients there."""
    cu = [0, 13, 13, 29, 38]
    H, Hk, d, bq, bk = 2, 1, 4, 8, 4
    q, k, v, go = _packed(cu, H, Hk, d, seed=3)
    scale = 0.5
    O, lse, _ = V.forward(q, k, v, cu, scale, bq, bk)
    tiles = [(-(-(b - a) // bq), -(-(b - a) // bk)) for a, b in zip(cu[:-1], cu[1:])]
    n_mask = sum(H * tr * tc for tr, tc in tiles)
    masks = np.random.default_rng(7).integers(0, 2, size=n_mask).astype(np.uint8)
    gq, gk, gv = V.backward(q, k, v, O, go, lse, cu, scale, masks, bq, bk)

    T = cu[-1]
    Mfull = np.zeros((H, T, T))
    off = 0
    for (a, b), (T_r, T_c) in zip(zip(cu[:-1], cu[1:]), tiles):
        n = b - a
        tm = masks[off:off + H * T_r * T_c].reshape(H, T_r, T_c)
        off += H * T_r * T_c
        r = np.arange(n)
        Mfull[:, a:a + n, a:a + n] = tm[:, r[:, None] // bq, r[None, :] // bk]
    qt, kt, vt, got = (torch.from_numpy(x) for x in (q, k, v, go))
    kk, vv = kt.repeat_interleave(H // Hk, 1), vt.repeat_interleave(H // Hk, 1)
    _, L_t, S_t = _block_diag_attention(qt, kt, vt, cu, scale)
    P = torch.exp(S_t - L_t[:, :, None]) * torch.from_numpy(Mfull)
    Ot = torch.from_numpy(O)
    Dr = torch.einsum("rhd,rhd->hr", got, Ot)
    GP = torch.einsum("rhd,chd->hrc", got, vv)
    GS = P * (GP - Dr[:, :, None])
    want_v = torch.einsum("hrc,rhd->chd", P, got).reshape(T, Hk, H // Hk, d).sum(2)
    want_k = scale * torch.einsum("hrc,rhd->chd", GS, qt).reshape(T, Hk, H // Hk, d).sum(2)
    want_q = scale * torch.einsum("hrc,chd->rhd", GS, kk)
    for mine, ref in ((gq, want_q), (gk, want_k), (gv, want_v)):
        assert np.allclose(mine, ref.numpy(), rtol=0, atol=1e-12)


def test_mask_of_equal_lengths_is_the_batched_mask():
    """Three sequences of one length pack exactly like a B = 3 batch, so the
    flat lists equal the fixed-length batched lists."""
    H, bq, bk, n = 2, 16, 8, 40
    cu = [0, n, 2 * n, 3 * n]
    q, k, v, _ = _packed(cu, H, H, 4, seed=5)
    q[:, 1] *= 3.0                                   # sharper rows on head 1
    scale = 0.9
    _, lse, stats = V.forward(q, k, v, cu, scale, bq, bk)
    got = V.mask_from_stats(stats.astype(np.float32), lse.astype(np.float32), cu, H, bq, bk, 0.2)
    T_r, T_c = -(-n // bq), -(-n // bk)
    ref = M.mask_from_stats(stats.astype(np.float32).reshape(3, H, T_c, T_r * bq),
                            lse.astype(np.float32).reshape(3, H, n), n, bq, bk, 0.2)
    for key in ("mask", "kv_idx", "kv_cnt", "q_idx", "q_cnt"):
        assert np.array_equal(got[key], np.asarray(ref[key]).reshape(-1)), key
    assert got["mask"].sum() < got["mask"].size      # something was skipped


def test_empty_sequences_change_nothing():
    H, Hk, d, bq, bk = 2, 2, 4, 8, 8
    cu_a = [0, 11, 30]
    cu_b = [0, 0, 11, 11, 11, 30, 30]
    q, k, v, go = _packed(cu_a, H, Hk, d, seed=2)
    Oa, la, sa = V.forward(q, k, v, cu_a, 0.5, bq, bk)
    Ob, lb, sb = V.forward(q, k, v, cu_b, 0.5, bq, bk)
    assert np.array_equal(Oa, Ob) and np.array_equal(la, lb) and np.array_equal(sa, sb)
    ga = V.backward(q, k, v, Oa, go, la, cu_a, 0.5)
    gb = V.backward(q, k, v, Ob, go, lb, cu_b, 0.5)
    for x, y in zip(ga, gb):
        assert np.array_equal(x, y)


def test_layout_totals_hand_count():
    # lengths 1, 128, 128, 128, 615, 0, 300; H = 4; 128 x 128 tiles:
    # T_r = T_c = 1, 1, 1, 1, 5, 0, 3 and n_pad = 128, 128, 128, 128, 640, 0, 384
    cu = [0, 1, 129, 257, 385, 1000, 1000, 1300]
    _, tot = V.layout(cu, 4, 128, 128)
    assert tot["total"] == 1300 and tot["lse"] == 5200
    assert tot["stats"] == 4 * (4 * 128 + 5 * 640 + 3 * 384)          # 19456
    assert tot["mask"] == 4 * (4 * 1 + 25 + 9) == tot["q_idx"]         # 152
    assert tot["kv_cnt"] == 4 * (4 + 5 + 3) == tot["q_cnt"]            # 48


def test_mask_of_ragged_lengths_is_each_sequences_own_mask():
    """With 16-row query tiles and 8-column key tiles the per-sequence blocks
    of kv_cnt (H*T_r) and q_cnt (H*T_c) differ in size: every block must hold
    the fixed-length lists of its own sequence's statistics."""
    H, bq, bk = 2, 16, 8
    cu = [0, 40, 41, 41, 70, 118]
    q, k, v, _ = _packed(cu, H, H, 4, seed=8)
    q[:, 0] *= 3.0
    _, lse, stats = V.forward(q, k, v, cu, 0.9, bq, bk)
    stats, lse = stats.astype(np.float32), lse.astype(np.float32)
    got = V.mask_from_stats(stats, lse, cu, H, bq, bk, 0.15)
    off = dict(stats=0, mask=0, kv_cnt=0, q_cnt=0)
    for a, b in zip(cu[:-1], cu[1:]):
        n = b - a
        T_r, T_c = -(-n // bq), -(-n // bk)
        if n:
            st = stats[off["stats"]:off["stats"] + H * T_c * T_r * bq].reshape(1, H, T_c, -1)
            ref = M.mask_from_stats(st, lse[H * a:H * b].reshape(1, H, n), n, bq, bk, 0.15)
            for key, o, size in (("mask", "mask", H * T_r * T_c),
                                 ("kv_idx", "mask", H * T_r * T_c),
                                 ("q_idx", "mask", H * T_c * T_r),
                                 ("kv_cnt", "kv_cnt", H * T_r), ("q_cnt", "q_cnt", H * T_c)):
                blk = got[key][off[o]:off[o] + size]
                assert np.array_equal(blk, np.asarray(ref[key]).reshape(-1)), (a, key)
        off["stats"] += H * T_c * T_r * bq
        off["mask"] += H * T_r * T_c
        off["kv_cnt"] += H * T_r
        off["q_cnt"] += H * T_c
    assert off["kv_cnt"] == got["kv_cnt"].size and off["q_cnt"] == got["q_cnt"].size
    assert 0 < got["mask"].sum() < got["mask"].size
