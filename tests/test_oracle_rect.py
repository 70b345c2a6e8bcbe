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
