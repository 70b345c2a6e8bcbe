"""GPU parity of rectangular attention (Nq queries, Nk keys): decoding against
a key/value cache (chapter 18 §18.8.2, FlashDecoding: a single query row per
head against a long cache, the key sequence split across CTAs and merged
through the log-sum-exp) and cross-attention.  With the causal mask the
queries are the last Nq positions.  The oracle's rectangular forward is the
reference; cases cover one and a few query rows, Nq > Nk, ragged Nk, cache
lengths per batch item (including 0), shared key/value heads, explicit and
planned key splits, and a 128K-key decode step on sampled heads.  O is held
to the flat 1e-2 except on rows that see fewer than 16 keys (N_q > N_k under
the causal mask, short caches), which are held to the worst case of the
kernel's two bf16 roundings (parity_util.assert_o)."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_10_gb300 import check_device_status, forward_rect, rect_split_count
from exact_tiled_attention_10_gb300.inputs import qkv, randn
from parity_util import assert_lse, assert_o, rounding_context, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(B, H, Hkv, Nq, Nk, d, causal, kv=None, num_splits=0, seed=3):
    q = randn((B, H, Nq, d), seed, device=DEV)
    k = randn((B, Hkv, Nk, d), seed + 1, device=DEV)
    v = randn((B, Hkv, Nk, d), seed + 2, device=DEV)
    kvd = None if kv is None else torch.tensor(kv, dtype=torch.int32, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = forward_rect(q, k, v, causal=causal, scale=scale, kv_lens=kvd, num_splits=num_splits)
    torch.cuda.synchronize()
    check_device_status()
    g = H // Hkv
    kvn = None if kv is None else np.asarray(kv, dtype=np.int32)
    kr, vr = np.repeat(to64(k), g, axis=1), np.repeat(to64(v), g, axis=1)
    run = lambda qq, vv: oracle.fwd_rect(qq, kr, vv, scale, causal=causal, kv_lens=kvn)
    ro, rl = run(to64(q), vr)
    nvis, absref = rounding_context(run, to64(q), vr)
    assert_o(to64(o), ro, nvis=nvis, absref=absref)
    assert_lse(to64(lse), rl)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(1, 1000), (4, 777), (64, 4096), (300, 1024)])
def test_rect_matches_oracle(d, causal, Nq, Nk):
    _case(2, 4, 4, Nq, Nk, d, causal, seed=Nq + Nk + d)


def test_grouped_heads_packed_across_tiles():
    """The query rows of the heads sharing a key/value head are processed as
    one block (row r is query r % Nq): causal limits that wrap inside a
    128-row tile."""
    _case(1, 4, 2, 300, 700, 128, True, seed=29)
    _case(2, 6, 2, 100, 5000, 64, True, kv=[4000, 5000], seed=31)
    _case(1, 8, 1, 33, 33, 128, True, seed=37)


def test_more_queries_than_keys_and_cache_lengths():
    _case(2, 2, 2, 500, 200, 128, True, seed=11)           # early rows see no key: O = 0, LSE = -inf
    _case(3, 4, 1, 3, 900, 128, True, kv=[0, 1, 900], seed=13)
    _case(2, 8, 2, 1, 3000, 64, False, kv=[1500, 2999], seed=17)


@pytest.mark.parametrize("num_splits", [1, 2, 7, 64])
def test_explicit_splits_agree(num_splits):
    _case(1, 2, 2, 2, 2049, 128, True, num_splits=num_splits, seed=19)


def test_planned_split_for_decode():
    assert rect_split_count(1, 8, 8, 1, 131072, 128, 0) > 1


def test_decode_128k_cache_sampled_heads():
    """One query per head (B = 1, H = 32, Hkv = 8) against a 131072-key cache:
    the planned split; two query heads of different groups against the oracle."""
    B, H, Hkv, Nq, Nk, d = 1, 32, 8, 1, 131072, 128
    q = randn((B, H, Nq, d), 23, device=DEV)
    k = randn((B, Hkv, Nk, d), 24, device=DEV)
    v = randn((B, Hkv, Nk, d), 25, device=DEV)
    o, lse = forward_rect(q, k, v, causal=True)
    torch.cuda.synchronize()
    check_device_status()
    g = H // Hkv
    for h in (0, 21):
        ro, rl = oracle.fwd_rect(to64(q[:, h:h + 1]), to64(k[:, h // g:h // g + 1]), to64(v[:, h // g:h // g + 1]),
                                 1.0 / math.sqrt(d), causal=True)
        assert_o(to64(o[:, h:h + 1]), ro)
        assert_lse(to64(lse[:, h:h + 1]), rl)


def _bwd_case(B, H, Hkv, Nq, Nk, d, causal, kv=None, seed=41, deterministic=False):
    from exact_tiled_attention_10_gb300 import backward_rect
    from parity_util import assert_grad
    q = randn((B, H, Nq, d), seed, device=DEV)
    k = randn((B, Hkv, Nk, d), seed + 1, device=DEV)
    v = randn((B, Hkv, Nk, d), seed + 2, device=DEV)
    do = randn((B, H, Nq, d), seed + 3, device=DEV)
    kvd = None if kv is None else torch.tensor(kv, dtype=torch.int32, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = forward_rect(q, k, v, causal=causal, scale=scale, kv_lens=kvd)
    dq, dk, dv = backward_rect(q, k, v, o, lse, do, causal=causal, scale=scale, kv_lens=kvd,
                               deterministic=deterministic)
    torch.cuda.synchronize()
    check_device_status()
    if deterministic:  # a second run agrees bit for bit
        again = backward_rect(q, k, v, o, lse, do, causal=causal, scale=scale, kv_lens=kvd, deterministic=True)
        torch.cuda.synchronize()
        for a, b in zip((dq, dk, dv), again):
            assert torch.equal(a, b)
    g = H // Hkv
    kvn = None if kv is None else np.asarray(kv, dtype=np.int32)
    r = oracle.bwd_rect(to64(q), np.repeat(to64(k), g, axis=1), np.repeat(to64(v), g, axis=1), to64(do), scale,
                        causal=causal, kv_lens=kvn)
    assert_grad(to64(dq), r["dq"], "dQ")
    assert_grad(to64(dk), r["dk"].reshape(B, Hkv, g, Nk, d).sum(axis=2), "dK")
    assert_grad(to64(dv), r["dv"].reshape(B, Hkv, g, Nk, d).sum(axis=2), "dV")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(200, 700), (700, 200), (64, 1000)])
def test_rect_backward_matches_oracle(d, causal, Nq, Nk):
    _bwd_case(2, 4, 2, Nq, Nk, d, causal, seed=Nq + 2 * Nk + d)


def test_rect_backward_with_cache_lengths_and_mqa():
    _bwd_case(3, 4, 1, 130, 390, 128, True, kv=[0, 100, 390], seed=53)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(200, 1700), (900, 300)])
def test_rect_backward_deterministic(d, causal, Nq, Nk):
    _bwd_case(2, 4, 2, Nq, Nk, d, causal, kv=[Nk, Nk // 3], seed=Nq + Nk + d + 5, deterministic=True)
