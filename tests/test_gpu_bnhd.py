"""GPU parity of the forward and backward on flash_attn_func's own layout
(chapter 18 §18.7.1: q is (batch, seqlen, nheads, headdim), k and v
(batch, seqlen_k, nheads_k, headdim), key/value heads broadcast when
nheads_k < nheads).  The oracle runs on the same tensors transposed to
[B, H, N, d]; LSE is [B, H, N].  At the long-head training shape the results
are compared with the [B, H, N, d] path on the transposed tensors."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_10_gb300 import (backward, backward_bnhd, check_device_status, forward,
                                           forward_bnhd)
from exact_tiled_attention_10_gb300.inputs import randn
from parity_util import O_TOL, assert_close_abs, assert_grad, assert_lse, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bhnd(x):
    """[B, N, H, d] -> [B, H, N, d] (float64 numpy)."""
    return np.ascontiguousarray(np.transpose(to64(x), (0, 2, 1, 3)))


@pytest.mark.parametrize("B,N,H,Hkv,d", [(2, 700, 4, 4, 128), (3, 300, 8, 2, 64), (1, 129, 4, 1, 128),
                                         (2, 1, 2, 2, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_bnhd_matches_oracle(B, N, H, Hkv, d, causal):
    seed = B * 7 + N + H + Hkv + d
    q = randn((B, N, H, d), seed, device=DEV)
    k = randn((B, N, Hkv, d), seed + 1, device=DEV)
    v = randn((B, N, Hkv, d), seed + 2, device=DEV)
    do = randn((B, N, H, d), seed + 3, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = forward_bnhd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = backward_bnhd(q, k, v, o, lse, do, causal=causal, scale=scale)
    torch.cuda.synchronize()
    check_device_status()
    g = H // Hkv
    kf, vf = np.repeat(_bhnd(k), g, axis=1), np.repeat(_bhnd(v), g, axis=1)
    ro, rl = oracle.fwd(_bhnd(q), kf, vf, scale, causal=causal)
    assert_close_abs(_bhnd(o), ro, O_TOL, "O")
    assert_lse(to64(lse), rl)
    r = oracle.bwd(_bhnd(q), kf, vf, _bhnd(do), scale, causal=causal)
    assert_grad(_bhnd(dq), r["dq"], "dQ")
    assert_grad(_bhnd(dk), r["dk"].reshape(B, Hkv, g, N, d).sum(axis=2), "dK")
    assert_grad(_bhnd(dv), r["dv"].reshape(B, Hkv, g, N, d).sum(axis=2), "dV")


def test_bnhd_long_head_agrees_with_the_bhnd_path():
    """B=2, N=4096, H=16, d=128, causal: both layouts against each other
    (each is within the oracle tolerances, so they agree within twice them)."""
    B, N, H, d = 2, 4096, 16, 128
    q, k, v, do = (randn((B, N, H, d), 1003 + i, device=DEV) for i in range(4))
    o, lse = forward_bnhd(q, k, v, causal=True)
    dq, dk, dv = backward_bnhd(q, k, v, o, lse, do, causal=True)
    t = [x.transpose(1, 2).contiguous() for x in (q, k, v, do)]
    o2, lse2 = forward(t[0], t[1], t[2], causal=True)
    g2 = backward(t[0], t[1], t[2], o2, lse2, t[3], causal=True)
    torch.cuda.synchronize()
    check_device_status()
    assert (o.transpose(1, 2).float() - o2.float()).abs().max().item() <= 2 * O_TOL
    assert (lse - lse2).abs().max().item() <= 2e-3
    for a, b in zip((dq, dk, dv), g2):
        a = a.transpose(1, 2).float()
        assert (a - b.float()).abs().max().item() <= 4e-2 * b.float().abs().max().item()


def test_bnhd_long_seq_agrees_with_the_bhnd_path():
    """B=1, N=16384, H=8, d=128, causal (the long-sequence shape): the
    [B, N, H, d] layout against the [B, H, N, d] path on the transposed
    tensors."""
    B, N, H, d = 1, 16384, 8, 128
    q, k, v, do = (randn((B, N, H, d), 1005 + i, device=DEV) for i in range(4))
    o, lse = forward_bnhd(q, k, v, causal=True)
    dq, dk, dv = backward_bnhd(q, k, v, o, lse, do, causal=True)
    t = [x.transpose(1, 2).contiguous() for x in (q, k, v, do)]
    o2, lse2 = forward(t[0], t[1], t[2], causal=True)
    g2 = backward(t[0], t[1], t[2], o2, lse2, t[3], causal=True)
    torch.cuda.synchronize()
    check_device_status()
    assert (o.transpose(1, 2).float() - o2.float()).abs().max().item() <= 2 * O_TOL
    assert (lse - lse2).abs().max().item() <= 2e-3
    for a, b in zip((dq, dk, dv), g2):
        a = a.transpose(1, 2).float()
        assert (a - b.float()).abs().max().item() <= 4e-2 * b.float().abs().max().item()
