"""Pins of the oracle's block-sparse mask (chapter 18 §18.8.1: for each query
block the list of key blocks to compute; blocks not listed are skipped, which
is the same as masking them).  The oracle takes the mask as a dense 0/1
matrix over bs x bs blocks.

Checked against: float64 torch autograd with the block mask expanded to an
element mask by a Kronecker product (index arithmetic independent of the
oracle), the all-ones mask (= no mask), the block-diagonal mask (= separate
attention problems on each block, run as separate oracle calls on slices),
an empty block row (fully masked rows: O = 0, LSE = -inf, zero gradients),
and central finite differences."""
import math

import numpy as np
import pytest
import torch

import oracle


def _autograd_elem(Q, K, V, G, scale, vis):
    q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
    vis = torch.tensor(vis, dtype=torch.bool)
    S = (scale * q @ k.transpose(-1, -2)).masked_fill(~vis, float("-inf"))
    rowany = vis.any(-1, keepdim=True)
    P = torch.softmax(S.masked_fill(~rowany, 0.0), dim=-1) * rowany
    O = P @ v
    O.backward(torch.tensor(G, dtype=torch.float64))
    return O.detach().numpy(), q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


def _elem(bm, bs, N):
    return np.kron(np.asarray(bm, dtype=bool), np.ones((bs, bs), dtype=bool))[:N, :N]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,bs", [(12, 4), (14, 4), (9, 3)])
def test_block_mask_against_autograd(causal, N, bs):
    rng = np.random.default_rng(N * 7 + bs + causal)
    B, H, d = 2, 2, 5
    nb = (N + bs - 1) // bs
    bm = rng.integers(0, 2, size=(nb, nb)).astype(np.uint8)
    bm[0, 0] = 1
    Q, K, V, dO = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    scale = 1 / math.sqrt(d)
    r = oracle.bwd(Q, K, V, dO, scale, causal=causal, block_mask=bm, block_size=bs)
    vis = _elem(bm, bs, N)
    if causal:
        vis = vis & np.tril(np.ones((N, N), dtype=bool))
    O, dq, dk, dv = _autograd_elem(Q, K, V, dO, scale, vis)
    for a, b in ((r["o"], O), (r["dq"], dq), (r["dk"], dk), (r["dv"], dv)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    o, lse = oracle.fwd(Q, K, V, scale, causal=causal, block_mask=bm, block_size=bs)
    np.testing.assert_allclose(o, O, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), ~vis.any(-1)[None, None].repeat(B, 0).repeat(H, 1))


def test_all_ones_block_mask_is_no_mask():
    rng = np.random.default_rng(3)
    Q, K, V, dO = (rng.standard_normal((1, 2, 10, 3)) for _ in range(4))
    for causal in (False, True):
        a = oracle.bwd(Q, K, V, dO, 0.5, causal=causal, kv_lens=np.array([7], np.int32))
        b = oracle.bwd(Q, K, V, dO, 0.5, causal=causal, kv_lens=np.array([7], np.int32),
                       block_mask=np.ones((4, 4)), block_size=3)
        for key in ("o", "lse", "dq", "dk", "dv"):
            np.testing.assert_array_equal(a[key], b[key])


def test_block_diagonal_mask_is_independent_blocks():
    """Diagonal block mask: each bs-row block attends only to its own keys, so
    every block is a separate attention problem of its own length."""
    rng = np.random.default_rng(4)
    N, bs = 11, 4
    Q, K, V, dO = (rng.standard_normal((1, 1, N, 3)) for _ in range(4))
    r = oracle.bwd(Q, K, V, dO, 0.8, block_mask=np.eye(3), block_size=bs)
    for a in range(0, N, bs):
        sl = slice(a, min(a + bs, N))
        p = oracle.bwd(Q[:, :, sl], K[:, :, sl], V[:, :, sl], dO[:, :, sl], 0.8)
        for key in ("o", "lse", "dq", "dk", "dv"):
            np.testing.assert_allclose(r[key][:, :, sl], p[key], rtol=0, atol=1e-14)


def test_empty_block_row_is_fully_masked():
    rng = np.random.default_rng(5)
    N, bs = 8, 4
    Q, K, V, dO = (rng.standard_normal((1, 1, N, 3)) for _ in range(4))
    bm = np.array([[1, 1], [0, 0]])
    r = oracle.bwd(Q, K, V, dO, 0.7, block_mask=bm, block_size=bs)
    assert np.all(r["o"][0, 0, 4:] == 0) and np.all(np.isneginf(r["lse"][0, 0, 4:]))
    assert np.all(r["dq"][0, 0, 4:] == 0)
    assert np.all(np.isfinite(r["lse"][0, 0, :4]))


@pytest.mark.parametrize("causal", [False, True])
def test_block_mask_finite_differences(causal):
    rng = np.random.default_rng(21)
    N, bs, d = 8, 3, 3
    Q, K, V, dO = (rng.standard_normal((1, 1, N, d)) for _ in range(4))
    bm = np.array([[1, 0, 1], [1, 1, 0], [0, 1, 1]])
    scale = 0.6
    r = oracle.bwd(Q, K, V, dO, scale, causal=causal, block_mask=bm, block_size=bs)
    h = 1e-6

    def loss(Qx, Kx, Vx):
        o, _ = oracle.fwd(Qx, Kx, Vx, scale, causal=causal, block_mask=bm, block_size=bs)
        return float(np.sum(o * dO))

    for name, X, grad in (("q", Q, r["dq"]), ("k", K, r["dk"]), ("v", V, r["dv"])):
        fd = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = {"q": (Xp, K, V), "k": (Q, Xp, V), "v": (Q, K, Xp)}[name]
            args_m = {"q": (Xm, K, V), "k": (Q, Xm, V), "v": (Q, K, Xm)}[name]
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.max(np.abs(fd - grad)) <= 1e-7 * max(1.0, np.max(np.abs(grad))), name


def test_block_mask_row_sampled_forms_match_full():
    rng = np.random.default_rng(35)
    N, d, bs = 40, 5, 8
    Q, K, V, dO = (rng.standard_normal((1, 1, N, d)) for _ in range(4))
    bm = rng.integers(0, 2, size=(5, 5))
    r = oracle.bwd(Q, K, V, dO, 0.4, causal=True, block_mask=bm, block_size=bs)
    rows = [0, 3, 8, 17, 31, 39]
    keys = [0, 7, 8, 22, 39]
    o_r, lse_r = oracle.fwd_rows(Q[0, 0], K[0, 0], V[0, 0], 0.4, True, N, rows, block_mask=bm, block_size=bs)
    np.testing.assert_allclose(o_r, r["o"][0, 0, rows], rtol=0, atol=1e-14)
    np.testing.assert_array_equal(np.isneginf(lse_r), np.isneginf(r["lse"][0, 0, rows]))
    g = oracle.bwd_rows(Q[0, 0], K[0, 0], V[0, 0], dO[0, 0], 0.4, True, N, rows, keys, block_mask=bm,
                        block_size=bs)
    np.testing.assert_allclose(g["dq"], r["dq"][0, 0, rows], rtol=0, atol=1e-13)
    np.testing.assert_allclose(g["dk"], r["dk"][0, 0, keys], rtol=0, atol=1e-13)
    np.testing.assert_allclose(g["dv"], r["dv"][0, 0, keys], rtol=0, atol=1e-13)
