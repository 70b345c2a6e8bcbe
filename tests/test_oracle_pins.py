"""Pins for the CPU oracle: values and properties fixed by the pages and by the
mathematics, independent of the oracle's own code.

Each test names the passage it follows.  Pages:
  FA2  = "解析 FlashAttention（4）：FlashAttention-v2" (FA-v2 analysis page)
  WIKI = "分块 Attention：重建概率，累计梯度" (attention-kernels wiki page)
  CH18 = "第18章 FlashAttention" (book chapter 18)
"""
import json
import math
import os

import mpmath
import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")
mpmath.mp.dps = 50


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# WIKI §02: six scores [1,2,-1,3,0,2.5]; online (any blocking) == full row.
# ---------------------------------------------------------------------------
def _six_score_problem(v2d=None):
    s = _load("wiki_six_scores.json")["scores"]
    N = len(s)
    # one query, six keys, scores realised as S = q.k with d = 1 and scale 1;
    # every query row is the same so the whole [N] row block carries the case
    q = np.ones((1, 1, N, 1))
    k = np.array(s, dtype=np.float64).reshape(1, 1, N, 1)
    return s, q, k


def test_six_scores_lse_and_probabilities_closed_form():
    s, q, k = _six_score_problem()
    N = len(s)
    # V = identity (d = N) makes O's row equal to the probability row P
    d = N
    qd = np.zeros((1, 1, N, d)); qd[..., 0] = 1.0
    kd = np.zeros((1, 1, N, d)); kd[..., 0] = np.array(s)
    v = np.eye(N).reshape(1, 1, N, d)
    o, lse = oracle.fwd(qd, kd, v, scale=1.0)
    Z = mpmath.fsum(mpmath.exp(mpmath.mpf(x)) for x in s)
    lse_exact = float(mpmath.log(Z))
    p_exact = [float(mpmath.exp(mpmath.mpf(x)) / Z) for x in s]
    assert abs(lse[0, 0, 0] - lse_exact) <= 1e-15 * abs(lse_exact)
    np.testing.assert_allclose(o[0, 0, 0], p_exact, rtol=1e-15, atol=0)
    # m = 3 and l = sum exp(s - 3): the running state after the last block
    l_exact = float(mpmath.fsum(mpmath.exp(mpmath.mpf(x) - 3) for x in s))
    assert abs(math.exp(lse[0, 0, 0] - 3.0) - l_exact) <= 1e-14 * l_exact


@pytest.mark.parametrize("Bc", [1, 2, 3, 4, 5, 6])
def test_six_scores_every_blocking_equals_full_row(Bc):
    s, _, _ = _six_score_problem()
    N, d = len(s), 2
    qd = np.zeros((1, 1, N, d)); qd[..., 0] = 1.0
    kd = np.zeros((1, 1, N, d)); kd[..., 0] = np.array(s)
    rng = np.random.default_rng(6)
    v = rng.standard_normal((1, 1, N, d))  # the page's 2-D values are not printed
    o_full, lse_full = oracle.fwd(qd, kd, v, scale=1.0)
    for Br in (1, 2, 6):
        o_t, lse_t = oracle.tiled_fwd(qd, kd, v, scale=1.0, Br=Br, Bc=Bc)
        np.testing.assert_allclose(o_t, o_full, rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(lse_t, lse_full, rtol=1e-15, atol=0)
    # and the value itself against 50-digit arithmetic
    Z = mpmath.fsum(mpmath.exp(mpmath.mpf(x)) for x in s)
    for t in range(d):
        exact = float(mpmath.fsum(mpmath.exp(mpmath.mpf(x)) * mpmath.mpf(float(v[0, 0, j, t]))
                                  for j, x in enumerate(s)) / Z)
        assert abs(o_full[0, 0, 0, t] - exact) <= 1e-14 * max(1.0, abs(exact))


# ---------------------------------------------------------------------------
# WIKI §04: five positions, 2-D Q/K/V/G, causal, 2x2 blocks.
# ---------------------------------------------------------------------------
def _five():
    g = _load("wiki_five_position.json")
    Q, K, V, G = (np.array(g[x], dtype=np.float64).reshape(1, 1, 5, 2) for x in "QKVG")
    return g, Q, K, V, G


def _mp_row(Q, K, i, scale, causal=True):
    """scores of row i and their mp log-sum-exp (closed form, 50 digits)."""
    js = [j for j in range(5) if (not causal or j <= i)]
    s = {j: scale * mpmath.fsum(mpmath.mpf(float(Q[0, 0, i, t])) * mpmath.mpf(float(K[0, 0, j, t]))
                                for t in range(2)) for j in js}
    Z = mpmath.fsum(mpmath.exp(x) for x in s.values())
    return s, mpmath.log(Z)


def test_five_position_visible_pair_count():
    g, *_ = _five()
    n = sum(1 for i in range(5) for j in range(5) if j <= i)
    assert n == g["visible_dot_products"] == 15


def test_five_position_closed_forms():
    g, Q, K, V, G = _five()
    scale = 1.0 / math.sqrt(g["d"])
    r = oracle.bwd(Q, K, V, G, scale, causal=True)
    # row 0 sees only key 0: O_0 = v_0, LSE_0 = S_00, dQ_0 = 0
    np.testing.assert_allclose(r["o"][0, 0, 0], V[0, 0, 0], rtol=0, atol=1e-15)
    s00 = (0.2 * 0.3 - 0.3 * 0.5) * scale
    assert abs(r["lse"][0, 0, 0] - s00) < 1e-15
    np.testing.assert_allclose(r["dq"][0, 0, 0], [0.0, 0.0], atol=1e-15)
    # key 4 is seen only by query 4: dV_4 = P_44 G_4
    s, L = _mp_row(Q, K, 4, scale)
    p44 = float(mpmath.exp(s[4] - L))
    np.testing.assert_allclose(r["dv"][0, 0, 4], p44 * G[0, 0, 4], rtol=1e-14, atol=1e-16)
    # every LSE and O row against 50-digit closed forms
    for i in range(5):
        s, L = _mp_row(Q, K, i, scale)
        assert abs(r["lse"][0, 0, i] - float(L)) < 1e-14
        for t in range(2):
            o_exact = float(mpmath.fsum(mpmath.exp(s[j] - L) * mpmath.mpf(float(V[0, 0, j, t])) for j in s))
            assert abs(r["o"][0, 0, i, t] - o_exact) < 1e-14


def test_five_position_blocked_backward_equals_full():
    g, Q, K, V, G = _five()
    scale = 1.0 / math.sqrt(g["d"])
    r = oracle.bwd(Q, K, V, G, scale, causal=True)
    o_t, lse_t = oracle.tiled_fwd(Q, K, V, scale, causal=True, Br=2, Bc=2)
    np.testing.assert_allclose(o_t, r["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse_t, r["lse"], rtol=0, atol=1e-14)
    dq, dk, dv = oracle.tiled_bwd(Q, K, V, o_t, lse_t, G, scale, causal=True, Br=2, Bc=2)
    for a, b in ((dq, r["dq"]), (dk, r["dk"]), (dv, r["dv"])):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)


def _autograd(Q, K, V, G, scale, causal, kv_lens=None):
    """Third implementation (tests only): float64 torch autograd of the
    materialised formula softmax(scale QK^T + M) V, with the gradient derived
    by autograd rather than written out."""
    q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
    B, H, N, d = Q.shape
    S = scale * q @ k.transpose(-1, -2)
    vis = torch.ones(B, 1, N, N, dtype=torch.bool)
    if causal:
        vis &= torch.ones(N, N, dtype=torch.bool).tril()
    if kv_lens is not None:
        cols = torch.arange(N)
        for b in range(B):
            vis[b] &= (cols < int(kv_lens[b]))[None, None, :]
    S = S.masked_fill(~vis, float("-inf"))
    rowany = vis.any(-1, keepdim=True)
    P = torch.softmax(S.masked_fill(~rowany, 0.0), dim=-1) * rowany
    O = P @ v
    O.backward(torch.tensor(G, dtype=torch.float64))
    return O.detach().numpy(), q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


def test_five_position_against_autograd():
    g, Q, K, V, G = _five()
    scale = 1.0 / math.sqrt(g["d"])
    r = oracle.bwd(Q, K, V, G, scale, causal=True)
    O, dq, dk, dv = _autograd(Q, K, V, G, scale, True)
    for a, b in ((r["o"], O), (r["dq"], dq), (r["dk"], dk), (r["dv"], dv)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------
# FA2 §3 / §5.3: N=4, d=3, Br=Bc=2 (symbolic on the page; seeded here).
# ---------------------------------------------------------------------------
def _n4_inputs():
    rng = np.random.default_rng(43)
    Q = rng.standard_normal((1, 1, 4, 3))
    K = rng.standard_normal((1, 1, 4, 3))
    V = rng.standard_normal((1, 1, 4, 3))
    dO = rng.standard_normal((1, 1, 4, 3))
    # make the running max RISE in block 2 for query 1 and STAY for query 2,
    # exercising both cases of the rescale of §3.3
    Q[0, 0, 0] = [1.0, 0.0, 0.0]
    Q[0, 0, 1] = [0.0, 1.0, 0.0]
    K[0, 0, :, 0] = [0.1, 0.2, 3.0, 0.3]   # query 1: block-2 key 3 wins
    K[0, 0, :, 1] = [2.5, 0.1, -0.4, 0.2]  # query 2: block-1 key 1 stays max
    return Q, K, V, dO


@pytest.mark.parametrize("causal", [False, True])
def test_n4_d3_blocking_equals_unblocked(causal):
    Q, K, V, dO = _n4_inputs()
    scale = 1.0 / math.sqrt(3)
    r = oracle.bwd(Q, K, V, dO, scale, causal=causal)
    o_t, lse_t = oracle.tiled_fwd(Q, K, V, scale, causal=causal, Br=2, Bc=2)
    np.testing.assert_allclose(o_t, r["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse_t, r["lse"], rtol=0, atol=1e-14)
    dq, dk, dv = oracle.tiled_bwd(Q, K, V, o_t, lse_t, dO, scale, causal=causal, Br=2, Bc=2)
    np.testing.assert_allclose(dq, r["dq"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk, r["dk"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv, r["dv"], rtol=0, atol=1e-14)
    # the constructed maxima really are where the comment says
    S = scale * Q[0, 0] @ K[0, 0].T
    assert np.argmax(S[0]) == 2 and np.argmax(S[1]) == 0


@pytest.mark.parametrize("Br,Bc", [(1, 3), (3, 2), (4, 4), (5, 3), (2, 7)])
@pytest.mark.parametrize("causal", [False, True])
def test_tiled_equals_naive_ragged_blocks(Br, Bc, causal):
    rng = np.random.default_rng(Br * 10 + Bc)
    B, H, N, d = 2, 2, 11, 4
    Q, K, V, dO = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    kv = np.array([7, 11], dtype=np.int32)
    scale = 0.7
    r = oracle.bwd(Q, K, V, dO, scale, causal=causal, kv_lens=kv)
    o_t, lse_t = oracle.tiled_fwd(Q, K, V, scale, causal=causal, kv_lens=kv, Br=Br, Bc=Bc)
    np.testing.assert_allclose(o_t, r["o"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse_t, r["lse"], rtol=0, atol=1e-13)
    dq, dk, dv = oracle.tiled_bwd(Q, K, V, o_t, lse_t, dO, scale, causal=causal, kv_lens=kv,
                                  Br=Br, Bc=Bc)
    for a, b in ((dq, r["dq"]), (dk, r["dk"]), (dv, r["dv"])):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# Finite differences of L = sum(O * dO) (an independent check of every
# gradient term: a dropped scale, a wrong sign or a transposed operand fails).
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal,kv", [(False, None), (True, None), (False, [5, 2]), (True, [3, 6])])
def test_finite_differences(causal, kv):
    rng = np.random.default_rng(7)
    B, H, N, d = 2, 1, 6, 3
    Q, K, V, dO = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    scale = 0.6
    kvn = None if kv is None else np.array(kv, dtype=np.int32)
    r = oracle.bwd(Q, K, V, dO, scale, causal=causal, kv_lens=kvn)
    h = 1e-6

    def loss(Qx, Kx, Vx):
        o, _ = oracle.fwd(Qx, Kx, Vx, scale, causal=causal, kv_lens=kvn)
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
        err = np.max(np.abs(fd - grad))
        assert err <= 1e-7 * max(1.0, np.max(np.abs(grad))), (name, err)


@pytest.mark.parametrize("causal,kv", [(False, None), (True, None), (False, [9, 4, 0]), (True, [12, 1, 7])])
def test_against_autograd_random(causal, kv):
    rng = np.random.default_rng(11)
    B, H, N, d = 3, 2, 12, 5
    Q, K, V, dO = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    scale = 1 / math.sqrt(d)
    kvn = None if kv is None else np.array(kv, dtype=np.int32)
    r = oracle.bwd(Q, K, V, dO, scale, causal=causal, kv_lens=kvn)
    O, dq, dk, dv = _autograd(Q, K, V, dO, scale, causal, kvn)
    for a, b in ((r["o"], O), (r["dq"], dq), (r["dk"], dk), (r["dv"], dv)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Identities and textbook special cases.
# ---------------------------------------------------------------------------
def test_rows_of_P_sum_to_one_and_D_identity():
    rng = np.random.default_rng(3)
    B, H, N, d = 2, 2, 9, 4
    Q, K, dO = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    V = np.ones((B, H, N, d))  # O = P 1 = row sums of P
    kv = np.array([9, 5], dtype=np.int32)
    for causal in (False, True):
        r = oracle.bwd(Q, K, V, dO, 0.5, causal=causal, kv_lens=kv)
        np.testing.assert_allclose(r["o"], 1.0, rtol=0, atol=1e-14)
    V = rng.standard_normal((B, H, N, d))
    for causal in (False, True):
        r = oracle.bwd(Q, K, V, dO, 0.5, causal=causal, kv_lens=kv)
        # FA2 §5.2: D_i = sum_j P_ij dP_ij equals rowsum(dO_i * O_i)
        np.testing.assert_allclose(r["D"], np.sum(dO * r["o"], -1), rtol=0, atol=1e-13)


def test_single_visible_key():
    rng = np.random.default_rng(5)
    B, H, N, d = 1, 2, 7, 3
    Q, K, V, dO = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    kv = np.array([1], dtype=np.int32)
    r = oracle.bwd(Q, K, V, dO, 0.8, causal=False, kv_lens=kv)
    np.testing.assert_allclose(r["o"], np.broadcast_to(V[:, :, :1], r["o"].shape), atol=1e-15)
    np.testing.assert_allclose(r["dq"], 0.0, atol=1e-15)
    np.testing.assert_allclose(r["dk"], 0.0, atol=1e-15)
    np.testing.assert_allclose(r["dv"][:, :, 0], dO.sum(2), atol=1e-14)
    np.testing.assert_allclose(r["dv"][:, :, 1:], 0.0, atol=0)
    # N = 1
    r1 = oracle.bwd(Q[:, :, :1], K[:, :, :1], V[:, :, :1], dO[:, :, :1], 0.8)
    np.testing.assert_allclose(r1["o"], V[:, :, :1], atol=1e-15)
    np.testing.assert_allclose(r1["dq"], 0.0, atol=1e-15)


def test_constant_scores_give_mean_of_visible_values():
    rng = np.random.default_rng(9)
    B, H, N, d = 1, 1, 8, 3
    Q, V = rng.standard_normal((B, H, N, d)), rng.standard_normal((B, H, N, d))
    K = np.zeros((B, H, N, d))
    o, lse = oracle.fwd(Q, K, V, 1.0, causal=True)
    for i in range(N):
        np.testing.assert_allclose(o[0, 0, i], V[0, 0, :i + 1].mean(0), atol=1e-15)
        assert abs(lse[0, 0, i] - math.log(i + 1)) < 1e-15
    o, lse = oracle.fwd(Q, K, V, 1.0, causal=False, kv_lens=np.array([5], dtype=np.int32))
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(V[0, 0, :5].mean(0), (N, d)), atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance(causal):
    """Adding one vector c to every key shifts each score row by a constant:
    P, O and dQ are unchanged (dQ_i changes by scale * c * sum_j dS_ij, which
    is 0 because every row of dS sums to zero) and dK is unchanged."""
    rng = np.random.default_rng(21)
    B, H, N, d = 1, 2, 10, 4
    Q, K, V, dO = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    c = rng.standard_normal(d)
    r0 = oracle.bwd(Q, K, V, dO, 0.5, causal=causal)
    r1 = oracle.bwd(Q, K + c, V, dO, 0.5, causal=causal)
    for key in ("o", "dq", "dk", "dv"):
        np.testing.assert_allclose(r1[key], r0[key], rtol=0, atol=1e-13)


def test_fully_masked_rows():
    """WIKI §04: a fully masked query row has O = 0, LSE = -inf, zero grads."""
    rng = np.random.default_rng(2)
    B, H, N, d = 2, 2, 6, 3
    Q, K, V, dO = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    kv = np.array([0, 6], dtype=np.int32)
    for causal in (False, True):
        r = oracle.bwd(Q, K, V, dO, 0.5, causal=causal, kv_lens=kv)
        assert np.all(r["o"][0] == 0.0)
        assert np.all(np.isneginf(r["lse"][0]))
        for key in ("dq", "dk", "dv"):
            assert np.all(r[key][0] == 0.0)
        assert np.all(np.isfinite(r["lse"][1]))
        o_t, lse_t = oracle.tiled_fwd(Q, K, V, 0.5, causal=causal, kv_lens=kv, Br=4, Bc=4)
        assert np.all(o_t[0] == 0.0) and np.all(np.isneginf(lse_t[0]))
        dq, dk, dv = oracle.tiled_bwd(Q, K, V, o_t, lse_t, dO, 0.5, causal=causal, kv_lens=kv, Br=4, Bc=4)
        assert np.all(dq[0] == 0.0) and np.all(dk[0] == 0.0) and np.all(dv[0] == 0.0)


# ---------------------------------------------------------------------------
# Row-sampled forms agree with the materialised ones.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal,kvl", [(False, 37), (True, 50), (True, 23), (False, 0)])
def test_row_sampled_forms_match_full(causal, kvl):
    rng = np.random.default_rng(31)
    N, d = 50, 8
    Q, K, V, dO = (rng.standard_normal((1, 1, N, d)) for _ in range(4))
    kv = np.array([kvl], dtype=np.int32)
    r = oracle.bwd(Q, K, V, dO, 0.35, causal=causal, kv_lens=kv)
    rows = [0, 1, 17, 36, 37, 49]
    keys = [0, 5, 22, 36, 49]
    o_r, lse_r = oracle.fwd_rows(Q[0, 0], K[0, 0], V[0, 0], 0.35, causal, kvl, rows)
    np.testing.assert_allclose(o_r, r["o"][0, 0, rows], rtol=0, atol=1e-14)
    np.testing.assert_array_equal(np.isneginf(lse_r), np.isneginf(r["lse"][0, 0, rows]))
    fin = np.isfinite(lse_r)
    np.testing.assert_allclose(lse_r[fin], r["lse"][0, 0, rows][fin], rtol=0, atol=1e-14)
    g = oracle.bwd_rows(Q[0, 0], K[0, 0], V[0, 0], dO[0, 0], 0.35, causal, kvl, rows, keys)
    np.testing.assert_allclose(g["dq"], r["dq"][0, 0, rows], rtol=0, atol=1e-13)
    np.testing.assert_allclose(g["dk"], r["dk"][0, 0, keys], rtol=0, atol=1e-13)
    np.testing.assert_allclose(g["dv"], r["dv"][0, 0, keys], rtol=0, atol=1e-13)
    np.testing.assert_allclose(g["D"], r["D"][0, 0], rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# FP8 E4M3 (CH18 §18.6.2).
# ---------------------------------------------------------------------------
def test_e4m3_closed_form_codes():
    assert oracle.e4m3_encode(1.0) == 0x38
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(-448.0) == 0xFE
    assert oracle.e4m3_encode(2.0 ** -9) == 0x01          # smallest subnormal
    assert oracle.e4m3_encode(2.0 ** -6) == 0x08          # smallest normal
    assert oracle.e4m3_encode(0.5) == 0x30
    assert oracle.e4m3_encode(1.0625) == 0x38             # tie 1 | 1.125 -> even (1.0)
    assert oracle.e4m3_encode(1.1875) == 0x3A             # tie 1.125 | 1.25 -> even (1.25)
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00         # tie 0 | 2^-9 -> even (0)
    assert oracle.e4m3_encode(1e6) == 0x7E                # saturation
    assert oracle.e4m3_encode(-1e30) == 0xFE
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert math.isnan(oracle.e4m3_decode(0x7F))


def test_e4m3_matches_torch_float8_in_range():
    """A library routine (torch's float8_e4m3fn cast, round-to-nearest-even)
    on every finite in-range input bucket, plus random fp32 values."""
    rng = np.random.default_rng(1)
    vals = [oracle.e4m3_decode(c) for c in range(0x7F)]
    mids = [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]
    xs = np.array(vals + mids + list(rng.uniform(-448, 448, 3000)) +
                  list(rng.standard_normal(3000) * 0.01), dtype=np.float32)
    xs = np.concatenate([xs, -xs])
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_encode(float(x)) for x in xs], dtype=np.uint8)
    # torch keeps the sign of zero like IEEE; so does the oracle
    np.testing.assert_array_equal(ours, ref)


def test_quantize_blocks_and_scales():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(1, 2, 150, 16, generator=g).to(torch.bfloat16)
    x[0, 1, 64:128] = 0  # an all-zero block takes scale 1
    codes, scales = oracle.quantize_fp8(x, blk=64)
    assert scales.shape == (1, 2, 3)
    xf = x.float().numpy()
    for h in range(2):
        for b in range(3):
            blk = xf[0, h, 64 * b:64 * (b + 1)]
            amax = np.float32(np.abs(blk).max())
            exp = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
            assert scales[0, h, b] == exp
    assert scales[0, 1, 1] == 1.0
    # the largest element of each non-zero block maps to +-448
    deq = oracle.dequantize_fp8(codes, scales)
    for h in range(2):
        for b in (0, 2):
            blk = xf[0, h, 64 * b:64 * (b + 1)]
            i = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
            assert abs(oracle.e4m3_decode(codes[0, h, 64 * b + i[0], i[1]])) == 448.0
    # E4M3 relative error bound: |x - deq| <= 2^-4 |x| for normal-range values
    rel = np.abs(deq - xf) / np.maximum(np.abs(xf), 1e-30)
    big = np.abs(xf) > 0.05
    assert np.all(rel[big] <= 2.0 ** -4 + 1e-7)
