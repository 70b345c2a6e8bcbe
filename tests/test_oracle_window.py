"""Pins of the oracle's sliding-window mask (chapter 18 §18.7.1,
flash_attn_func's window_size=(left, right): key j is visible to query i only
if i - left <= j <= i + right, -1 meaning no bound on that side).

The window is checked against things other than the oracle itself: float64
torch autograd of the materialised formula with the window written as an
explicit additive mask (built here from index arithmetic, gradients derived
by autograd), the window (0, 0) closed form, the causal mask as window
(-1, 0), windows wider than the sequence, and central finite differences.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _autograd_window(Q, K, V, G, scale, causal, wl, wr, kv_lens=None):
    """float64 autograd of softmax(scale Q K^T + M) V, M = -inf outside the
    window / causal / key-padding pattern; fully masked rows give O = 0."""
    q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
    B, H, N, d = Q.shape
    i = torch.arange(N)[:, None]
    j = torch.arange(N)[None, :]
    vis = torch.ones(N, N, dtype=torch.bool)
    if causal:
        vis &= j <= i
    if wl >= 0:
        vis &= j >= i - wl
    if wr >= 0:
        vis &= j <= i + wr
    vis = vis[None, None].expand(B, 1, N, N).clone()
    if kv_lens is not None:
        for b in range(B):
            vis[b] &= (torch.arange(N) < int(kv_lens[b]))[None, None, :]
    S = (scale * q @ k.transpose(-1, -2)).masked_fill(~vis, float("-inf"))
    rowany = vis.any(-1, keepdim=True)
    P = torch.softmax(S.masked_fill(~rowany, 0.0), dim=-1) * rowany
    O = P @ v
    O.backward(torch.tensor(G, dtype=torch.float64))
    return O.detach().numpy(), q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("causal,wl,wr,kv", [
    (False, 3, 2, None), (False, 0, 5, None), (False, 7, -1, None), (False, -1, 1, [13, 4]),
    (True, 4, -1, None), (True, 2, 3, [9, 13]), (False, 2, 2, [0, 6]), (True, 0, 0, None),
])
def test_window_against_autograd(causal, wl, wr, kv):
    rng = np.random.default_rng(101)
    B, H, N, d = 2, 2, 13, 5
    Q, K, V, dO = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    scale = 1 / math.sqrt(d)
    kvn = None if kv is None else np.array(kv, dtype=np.int32)
    r = oracle.bwd(Q, K, V, dO, scale, causal=causal, kv_lens=kvn, window=(wl, wr))
    O, dq, dk, dv = _autograd_window(Q, K, V, dO, scale, causal, wl, wr, kvn)
    for a, b in ((r["o"], O), (r["dq"], dq), (r["dk"], dk), (r["dv"], dv)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    o, lse = oracle.fwd(Q, K, V, scale, causal=causal, kv_lens=kvn, window=(wl, wr))
    np.testing.assert_allclose(o, O, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(r["lse"]))


def test_window_zero_zero_closed_form():
    """Each query sees only its own key: O_i = v_i, LSE_i = scale q_i.k_i,
    P_ii = 1 so dS = 0 (dQ = dK = 0) and dV_i = dO_i."""
    rng = np.random.default_rng(5)
    B, H, N, d = 1, 3, 10, 4
    Q, K, V, dO = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    r = oracle.bwd(Q, K, V, dO, 0.7, window=(0, 0))
    np.testing.assert_allclose(r["o"], V, rtol=0, atol=1e-15)
    np.testing.assert_allclose(r["lse"], 0.7 * np.sum(Q * K, axis=-1), rtol=0, atol=1e-14)
    assert np.max(np.abs(r["dq"])) <= 1e-15 and np.max(np.abs(r["dk"])) <= 1e-15
    np.testing.assert_allclose(r["dv"], dO, rtol=0, atol=1e-15)


def test_window_left_unbounded_right_zero_is_causal():
    rng = np.random.default_rng(6)
    Q, K, V, dO = (rng.standard_normal((2, 1, 11, 3)) for _ in range(4))
    a = oracle.bwd(Q, K, V, dO, 0.5, causal=True)
    b = oracle.bwd(Q, K, V, dO, 0.5, causal=False, window=(-1, 0))
    for key in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_array_equal(a[key], b[key])


def test_window_wider_than_sequence_is_no_window():
    rng = np.random.default_rng(8)
    N = 9
    Q, K, V, dO = (rng.standard_normal((1, 2, N, 3)) for _ in range(4))
    for causal in (False, True):
        a = oracle.bwd(Q, K, V, dO, 0.5, causal=causal)
        b = oracle.bwd(Q, K, V, dO, 0.5, causal=causal, window=(N - 1, N - 1))
        for key in ("o", "lse", "dq", "dk", "dv"):
            np.testing.assert_array_equal(a[key], b[key])


@pytest.mark.parametrize("causal,wl,wr", [(False, 1, 2), (True, 2, -1), (False, 0, 3)])
def test_window_finite_differences(causal, wl, wr):
    rng = np.random.default_rng(17)
    B, H, N, d = 1, 1, 7, 3
    Q, K, V, dO = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    scale = 0.6
    r = oracle.bwd(Q, K, V, dO, scale, causal=causal, window=(wl, wr))
    h = 1e-6

    def loss(Qx, Kx, Vx):
        o, _ = oracle.fwd(Qx, Kx, Vx, scale, causal=causal, window=(wl, wr))
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


@pytest.mark.parametrize("causal,wl,wr,kvl", [(False, 5, 3, 40), (True, 9, -1, 50), (False, -1, 0, 23)])
def test_window_row_sampled_forms_match_full(causal, wl, wr, kvl):
    rng = np.random.default_rng(33)
    N, d = 50, 6
    Q, K, V, dO = (rng.standard_normal((1, 1, N, d)) for _ in range(4))
    kv = np.array([kvl], dtype=np.int32)
    r = oracle.bwd(Q, K, V, dO, 0.4, causal=causal, kv_lens=kv, window=(wl, wr))
    rows = [0, 1, 17, 36, 45, 49]
    keys = [0, 5, 22, 39, 49]
    o_r, lse_r = oracle.fwd_rows(Q[0, 0], K[0, 0], V[0, 0], 0.4, causal, kvl, rows, window=(wl, wr))
    np.testing.assert_allclose(o_r, r["o"][0, 0, rows], rtol=0, atol=1e-14)
    np.testing.assert_array_equal(np.isneginf(lse_r), np.isneginf(r["lse"][0, 0, rows]))
    g = oracle.bwd_rows(Q[0, 0], K[0, 0], V[0, 0], dO[0, 0], 0.4, causal, kvl, rows, keys, window=(wl, wr))
    np.testing.assert_allclose(g["dq"], r["dq"][0, 0, rows], rtol=0, atol=1e-13)
    np.testing.assert_allclose(g["dk"], r["dk"][0, 0, keys], rtol=0, atol=1e-13)
    np.testing.assert_allclose(g["dv"], r["dv"][0, 0, keys], rtol=0, atol=1e-13)
