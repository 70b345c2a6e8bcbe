"""GPU parity of shared key/value heads (chapter 18 §18.7.1: with fewer
key/value heads than query heads, K and V are broadcast over the head
dimension; grouped-query attention, multi-query for one key/value head).
The oracle has no such notion, so the reference broadcasts K and V to every
query head (K_h = K[h // group]) and runs the ordinary oracle; the gradient
of a broadcast is the sum over the heads it feeds, so dK, dV of a key/value
head are the oracle's dK, dV summed over its group."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_10_gb300 import backward, check_device_status, forward
from exact_tiled_attention_10_gb300.inputs import qkv
from parity_util import O_TOL, assert_close_abs, assert_grad, assert_lse, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _gqa_case(B, H, Hkv, N, d, causal, kv=None, seed=3):
    q, _, _, do = qkv(B, H, N, d, seed, device=DEV)
    _, k, v = qkv(B, Hkv, N, d, seed + 50, device=DEV, with_dout=False)
    kvd = None if kv is None else torch.tensor(kv, dtype=torch.int32, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = forward(q, k, v, causal=causal, scale=scale, kv_lens=kvd)
    dq, dk, dv = backward(q, k, v, o, lse, do, causal=causal, scale=scale, kv_lens=kvd)
    torch.cuda.synchronize()
    check_device_status()
    assert dk.shape == (B, Hkv, N, d) and dv.shape == (B, Hkv, N, d)
    g = H // Hkv
    k_full = np.repeat(to64(k), g, axis=1)  # head h <- key/value head h // g
    v_full = np.repeat(to64(v), g, axis=1)
    kvn = None if kv is None else np.asarray(kv, dtype=np.int32)
    ref = oracle.bwd(to64(q), k_full, v_full, to64(do), scale, causal=causal, kv_lens=kvn)
    assert_close_abs(to64(o), ref["o"], O_TOL, "O")
    assert_lse(to64(lse), ref["lse"])
    assert_grad(to64(dq), ref["dq"], "dQ")
    dk_ref = ref["dk"].reshape(B, Hkv, g, N, d).sum(axis=2)
    dv_ref = ref["dv"].reshape(B, Hkv, g, N, d).sum(axis=2)
    assert_grad(to64(dk), dk_ref, "dK (group sum)")
    assert_grad(to64(dv), dv_ref, "dV (group sum)")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv", [(4, 2), (4, 1), (6, 3)])
def test_shared_kv_heads_match_broadcast_oracle(d, causal, H, Hkv):
    _gqa_case(2, H, Hkv, 300, d, causal, seed=H * 10 + Hkv + d)


def test_shared_kv_heads_with_key_padding():
    _gqa_case(3, 4, 2, 257, 128, True, kv=[0, 100, 257], seed=9)


def test_shared_kv_heads_equal_to_all_heads_is_the_plain_path():
    q, k, v = qkv(1, 4, 520, 128, 21, device=DEV, with_dout=False)
    o1, l1 = forward(q, k, v, causal=True)
    # the same K, V given as 2 shared heads each used by 2 query heads
    k2 = k[:, ::2].contiguous()
    v2 = v[:, ::2].contiguous()
    o2, l2 = forward(q, k2, v2, causal=True)
    o3, l3 = forward(q, k2.repeat_interleave(2, dim=1), v2.repeat_interleave(2, dim=1), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o2, o3) and torch.equal(l2, l3)
    assert torch.equal(o1[:, ::2], o2[:, ::2])
