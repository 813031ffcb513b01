"""Pins for the oracle's (masked) attention backward (CPU only).

* Dense case: central finite differences of L = sum(G_O * O(Q, K, V)) and
  fp64 torch autograd of softmax attention.
* Masked case: the masked gradients are linear in the tile mask (G_V, G_S,
  G_Q, G_K are all linear in M; D does not depend on M), so the gradients of
  a partition of the tiles must add up to the dense gradients pinned above; a
  single kept tile (i, j) must leave G_Q nonzero only in query tile i and
  G_K/G_V nonzero only in key tile j (catches a transposed mask).
"""
import numpy as np
import pytest
import torch

from oracle import attention as A


def _rand(shape, seed, s=1.0):
    return s * np.random.default_rng(seed).standard_normal(shape)


def _problem(B=1, n=12, H=2, Hk=1, d=4, seed=0):
    q = _rand((B, n, H, d), seed + 1, 1.5)
    k = _rand((B, n, Hk, d), seed + 2, 1.5)
    v = _rand((B, n, Hk, d), seed + 3)
    go = _rand((B, n, H, d), seed + 4)
    return q, k, v, go


def _loss(q, k, v, go, scale):
    O, _, _ = A.forward(q, k, v, scale)
    return float(np.sum(go * O))


@pytest.mark.parametrize("H,Hk", [(1, 1), (2, 1)])
def test_dense_gradient_matches_finite_differences(H, Hk):
    q, k, v, go = _problem(n=9, H=H, Hk=Hk, d=3, seed=H)
    scale = 0.7
    O, L, _ = A.forward(q, k, v, scale)
    gq, gk, gv = A.backward(q, k, v, O, go, L, scale)
    h = 1e-6
    for name, x, g in (("q", q, gq), ("k", k, gk), ("v", v, gv)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], go, scale)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], go, scale)
            fd[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(fd - g) / np.linalg.norm(fd)
        assert err < 1e-6, (name, err)


def test_dense_gradient_matches_torch_autograd_fp64():
    B, n, H, Hk, d = 2, 37, 4, 2, 8
    q, k, v, go = _problem(B, n, H, Hk, d, seed=5)
    scale = 0.3
    O, L, _ = A.forward(q, k, v, scale)
    gq, gk, gv = A.backward(q, k, v, O, go, L, scale)
    tq, tk, tv = (torch.from_numpy(x).clone().requires_grad_(True) for x in (q, k, v))
    G = H // Hk
    kk = tk.repeat_interleave(G, dim=2)
    vv = tv.repeat_interleave(G, dim=2)
    S = scale * torch.einsum("bnhd,bmhd->bhnm", tq, kk)
    O_t = torch.einsum("bhnm,bmhd->bnhd", torch.softmax(S, dim=-1), vv)
    O_t.backward(torch.from_numpy(go))
    for mine, ref in ((gq, tq.grad), (gk, tk.grad), (gv, tv.grad)):
        assert np.allclose(mine, ref.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(O, O_t.detach().numpy(), atol=1e-13)


def test_all_ones_mask_is_bitwise_dense():
    q, k, v, go = _problem(n=40, H=2, Hk=2, d=8, seed=9)
    scale = 0.35
    O, L, _ = A.forward(q, k, v, scale)
    dense = A.backward(q, k, v, O, go, L, scale)
    ones = np.ones((1, 2, 3, 3), dtype=np.uint8)
    masked = A.backward(q, k, v, O, go, L, scale, ones, 16, 16)
    for a, b in zip(dense, masked):
        assert np.array_equal(a, b)


def test_masked_gradients_are_linear_in_the_mask():
    n, bq, bk = 50, 16, 8
    q, k, v, go = _problem(n=n, H=2, Hk=1, d=8, seed=11)
    scale = 0.4
    O, L, _ = A.forward(q, k, v, scale)
    dense = A.backward(q, k, v, O, go, L, scale)
    T_r, T_c = -(-n // bq), -(-n // bk)
    part = np.random.default_rng(3).integers(0, 3, size=(1, 2, T_r, T_c))
    total = [np.zeros_like(x) for x in dense]
    for p in range(3):
        m = (part == p).astype(np.uint8)
        g = A.backward(q, k, v, O, go, L, scale, m, bq, bk)
        total = [t + x for t, x in zip(total, g)]
    for t, x in zip(total, dense):
        assert np.allclose(t, x, rtol=0, atol=1e-12)


def test_single_kept_tile_support():
    n, bq, bk = 48, 16, 16
    q, k, v, go = _problem(n=n, H=1, Hk=1, d=4, seed=13)
    scale = 0.5
    O, L, _ = A.forward(q, k, v, scale)
    m = np.zeros((1, 1, 3, 3), dtype=np.uint8)
    m[0, 0, 0, 2] = 1                      # query tile 0 x key tile 2
    gq, gk, gv = A.backward(q, k, v, O, go, L, scale, m, bq, bk)
    assert np.all(gq[0, 16:] == 0) and np.any(gq[0, :16] != 0)
    assert np.all(gk[0, :32] == 0) and np.any(gk[0, 32:] != 0)
    assert np.all(gv[0, :32] == 0) and np.any(gv[0, 32:] != 0)


def test_row_and_column_slices_agree_with_full():
    n, bq, bk = 70, 32, 32
    q, k, v, go = _problem(n=n, H=1, Hk=1, d=8, seed=17)
    scale = 0.45
    O, L, _ = A.forward(q, k, v, scale)
    m = np.random.default_rng(5).integers(0, 2, size=(1, 1, 3, 3)).astype(np.uint8)
    gq, gk, gv = A.backward(q, k, v, O, go, L, scale, m, bq, bk)
    rows = np.array([3, 40, 69])
    a, _, _ = A.backward_head(q[0, :, 0], k[0, :, 0], v[0, :, 0], O[0, :, 0], go[0, :, 0],
                              L[0, 0], scale, m[0, 0], bq, bk, rows=rows)
    assert np.allclose(a, gq[0, rows, 0], atol=1e-13)
    cols = np.arange(32, 64)
    _, b, c = A.backward_head(q[0, :, 0], k[0, :, 0], v[0, :, 0], O[0, :, 0], go[0, :, 0],
                              L[0, 0], scale, m[0, 0], bq, bk, cols=cols)
    assert np.allclose(b, gk[0, cols, 0], atol=1e-13)
    assert np.allclose(c, gv[0, cols, 0], atol=1e-13)


def test_stored_output_is_bf16_round_to_nearest_even():
    # 1 + 2^-8 lies exactly between two bf16 values (spacing 2^-7): ties go to
    # the even mantissa (1.0); 1 + 3*2^-8 rounds up to 1 + 2^-6.
    x = np.array([[1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -3.0e38, 0.1]])
    y = A.as_stored_output(x)
    assert y[0, 0] == 1.0 and y[0, 1] == 1.0 + 2.0 ** -6
    assert abs(y[0, 3] - 0.1) <= 0.1 * 2.0 ** -9


@pytest.mark.parametrize("window", [0, 6])
def test_causal_window_gradient_matches_torch_autograd(window):
    B, n, H, Hk, d = 1, 23, 2, 1, 4
    q, k, v, go = _problem(B, n, H, Hk, d, seed=41)
    scale = 0.5
    O, L, _ = A.forward(q, k, v, scale, causal=True, window=window)
    gq, gk, gv = A.backward(q, k, v, O, go, L, scale, causal=True, window=window)
    tq, tk, tv = (torch.from_numpy(x).clone().requires_grad_(True) for x in (q, k, v))
    r = torch.arange(n)[:, None]
    c = torch.arange(n)[None, :]
    m = (c <= r) & ((c > r - window) if window else torch.ones_like(c <= r))
    S = scale * torch.einsum("bnhd,bmhd->bhnm", tq, tk.repeat_interleave(2, dim=2))
    S = S.masked_fill(~m, float("-inf"))
    O_t = torch.einsum("bhnm,bmhd->bnhd", torch.softmax(S, dim=-1), tv.repeat_interleave(2, dim=2))
    O_t.backward(torch.from_numpy(go))
    for mine, ref in ((gq, tq.grad), (gk, tk.grad), (gv, tv.grad)):
        assert np.allclose(mine, ref.numpy(), rtol=0, atol=1e-12)
