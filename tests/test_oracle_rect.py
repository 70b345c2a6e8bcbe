"""Pins of the oracle's rectangular forward (Nq queries, Nk keys; chapter 18
§18.8.2: a decode step's query is [b, n_q, d] against a long key/value
cache; with the causal mask the queries are the last Nq positions).

Checked against: the square oracle when Nq = Nk (exactly), the last Nq rows
of the square causal oracle run on the full Nk-row sequence (exactly: the
same keys in the same order), float64 torch softmax with an explicit
bottom-right mask, and the one-query closed form."""
import math

import numpy as np
import pytest
import torch

import oracle


def test_square_shape_is_the_square_oracle():
    rng = np.random.default_rng(1)
    q, k, v = (rng.standard_normal((2, 2, 11, 4)) for _ in range(3))
    for causal in (False, True):
        kv = np.array([11, 6], np.int32)
        a = oracle.fwd(q, k, v, 0.4, causal=causal, kv_lens=kv)
        b = oracle.fwd_rect(q, k, v, 0.4, causal=causal, kv_lens=kv)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("Nq", [1, 3, 8])
def test_causal_queries_are_the_last_positions(Nq):
    rng = np.random.default_rng(2 + Nq)
    Nk = 13
    qf, k, v = (rng.standard_normal((1, 3, Nk, 5)) for _ in range(3))
    full_o, full_lse = oracle.fwd(qf, k, v, 0.3, causal=True)
    o, lse = oracle.fwd_rect(qf[:, :, Nk - Nq:], k, v, 0.3, causal=True)
    np.testing.assert_array_equal(o, full_o[:, :, Nk - Nq:])
    np.testing.assert_array_equal(lse, full_lse[:, :, Nk - Nq:])


@pytest.mark.parametrize("causal,kv", [(False, None), (True, None), (False, [17, 5]), (True, [9, 20])])
def test_rect_against_torch(causal, kv):
    rng = np.random.default_rng(7)
    B, H, Nq, Nk, d = 2, 2, 6, 20, 8
    q = rng.standard_normal((B, H, Nq, d))
    k, v = (rng.standard_normal((B, H, Nk, d)) for _ in range(2))
    scale = 1 / math.sqrt(d)
    kvn = None if kv is None else np.array(kv, np.int32)
    o, lse = oracle.fwd_rect(q, k, v, scale, causal=causal, kv_lens=kvn)
    S = torch.tensor(q) @ torch.tensor(k).transpose(-1, -2) * scale
    i = torch.arange(Nq)[:, None]
    j = torch.arange(Nk)[None, :]
    vis = torch.ones(B, 1, Nq, Nk, dtype=torch.bool)
    if causal:
        vis &= (j <= i + (Nk - Nq))
    if kvn is not None:
        for b in range(B):
            vis[b] &= (torch.arange(Nk) < int(kvn[b]))
    S = S.masked_fill(~vis, float("-inf"))
    ref_lse = torch.logsumexp(S, dim=-1)
    ref_o = torch.softmax(S, dim=-1) @ torch.tensor(v)
    np.testing.assert_allclose(o, ref_o.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=0, atol=1e-12)


def test_single_query_closed_form():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((1, 1, 1, 6))
    k, v = (rng.standard_normal((1, 1, 50, 6)) for _ in range(2))
    o, lse = oracle.fwd_rect(q, k, v, 0.5, causal=True)  # one query at the last position sees every key
    s = 0.5 * (k[0, 0] @ q[0, 0, 0])
    m = s.max()
    L = m + math.log(np.sum(np.exp(s - m)))
    assert abs(lse[0, 0, 0] - L) <= 1e-13
    np.testing.assert_allclose(o[0, 0, 0], np.exp(s - L) @ v[0, 0], rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal,kv,Nq,Nk", [(False, None, 5, 12), (True, None, 5, 12), (True, [9, 12], 4, 12),
                                              (True, None, 9, 6), (False, [3, 7], 7, 7)])
def test_rect_backward_against_autograd(causal, kv, Nq, Nk):
    rng = np.random.default_rng(Nq * 3 + Nk + causal)
    B, H, d = 2, 2, 4
    q, dO = (rng.standard_normal((B, H, Nq, d)) for _ in range(2))
    k, v = (rng.standard_normal((B, H, Nk, d)) for _ in range(2))
    scale = 0.7
    kvn = None if kv is None else np.array(kv, np.int32)
    r = oracle.bwd_rect(q, k, v, dO, scale, causal=causal, kv_lens=kvn)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    i = torch.arange(Nq)[:, None]
    j = torch.arange(Nk)[None, :]
    vis = torch.ones(B, 1, Nq, Nk, dtype=torch.bool)
    if causal:
        vis &= (j <= i + (Nk - Nq))
    if kvn is not None:
        for b in range(B):
            vis[b] &= (torch.arange(Nk) < int(kvn[b]))
    S = (scale * tq @ tk.transpose(-1, -2)).masked_fill(~vis, float("-inf"))
    rowany = vis.any(-1, keepdim=True)
    P = torch.softmax(S.masked_fill(~rowany, 0.0), dim=-1) * rowany
    (P @ tv).backward(torch.tensor(dO))
    for a, b in ((r["dq"], tq.grad), (r["dk"], tk.grad), (r["dv"], tv.grad)):
        np.testing.assert_allclose(a, b.numpy(), rtol=0, atol=1e-12)


def test_rect_backward_square_is_the_square_oracle():
    rng = np.random.default_rng(41)
    q, k, v, dO = (rng.standard_normal((1, 2, 10, 3)) for _ in range(4))
    for causal in (False, True):
        a = oracle.bwd(q, k, v, dO, 0.5, causal=causal)
        b = oracle.bwd_rect(q, k, v, dO, 0.5, causal=causal)
        for key in ("dq", "dk", "dv"):
            np.testing.assert_array_equal(a[key], b[key])


def test_rect_backward_finite_differences():
    rng = np.random.default_rng(43)
    Nq, Nk, d = 3, 7, 3
    q, dO = (rng.standard_normal((1, 1, Nq, d)) for _ in range(2))
    k, v = (rng.standard_normal((1, 1, Nk, d)) for _ in range(2))
    r = oracle.bwd_rect(q, k, v, dO, 0.6, causal=True)
    h = 1e-6

    def loss(qx, kx, vx):
        o, _ = oracle.fwd_rect(qx, kx, vx, 0.6, causal=True)
        return float(np.sum(o * dO))

    for name, X, grad in (("q", q, r["dq"]), ("k", k, r["dk"]), ("v", v, r["dv"])):
        fd = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = {"q": (Xp, k, v), "k": (q, Xp, v), "v": (q, k, Xp)}[name]
            args_m = {"q": (Xm, k, v), "k": (q, Xm, v), "v": (q, k, Xm)}[name]
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.max(np.abs(fd - grad)) <= 1e-7 * max(1.0, np.max(np.abs(grad))), name
