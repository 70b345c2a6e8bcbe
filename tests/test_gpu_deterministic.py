"""GPU checks of the deterministic backward (flash_attn_func's `deterministic`
flag, chapter 18 §18.7.1): parity with the fp64 oracle's gradients ([FA2]
§5.4 Algorithm 2), and bitwise-identical dQ, dK, dV over repeated runs, with
the workspace refilled with garbage in between and with another kernel
running beside it on a second stream."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_10_gb300 import (backward, backward_bnhd, backward_varlen, check_device_status, forward,
                                           forward_bnhd, forward_varlen, load_library, attn_params,
                                           FA_LAYOUT_PACKED)
from exact_tiled_attention_10_gb300.inputs import qkv, randn
from parity_util import assert_grad, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(B, H, Hkv, N, d, seed):
    q = randn((B, H, N, d), seed, device=DEV)
    k = randn((B, Hkv, N, d), seed + 1, device=DEV)
    v = randn((B, Hkv, N, d), seed + 2, device=DEV)
    do = randn((B, H, N, d), seed + 3, device=DEV)
    return q, k, v, do


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv,N,kv", [(4, 4, 700, None), (4, 2, 300, [300, 129]), (4, 1, 520, [0, 333])])
def test_deterministic_matches_oracle(d, causal, H, Hkv, N, kv):
    B = 2
    q, k, v, do = _inputs(B, H, Hkv, N, d, seed=N + d + H * Hkv)
    kvd = None if kv is None else torch.tensor(kv, dtype=torch.int32, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = forward(q, k, v, causal=causal, scale=scale, kv_lens=kvd)
    dq, dk, dv = backward(q, k, v, o, lse, do, causal=causal, scale=scale, kv_lens=kvd, deterministic=True)
    torch.cuda.synchronize()
    check_device_status()
    g = H // Hkv
    kvn = None if kv is None else np.asarray(kv, dtype=np.int32)
    r = oracle.bwd(to64(q), np.repeat(to64(k), g, axis=1), np.repeat(to64(v), g, axis=1), to64(do), scale,
                   causal=causal, kv_lens=kvn)
    assert_grad(to64(dq), r["dq"], "dQ")
    assert_grad(to64(dk), r["dk"].reshape(B, Hkv, g, N, d).sum(axis=2), "dK")
    assert_grad(to64(dv), r["dv"].reshape(B, Hkv, g, N, d).sum(axis=2), "dV")


def attn_bwd_workspace_size(**fields) -> int:
    """Workspace bytes the backward needs for these parameters (fa_attn_bwd_workspace_size)."""
    import ctypes
    p = attn_params(**fields)
    return int(load_library().fa_attn_bwd_workspace_size(ctypes.byref(p)))


def _repeat_bitwise(B, H, Hkv, N, d, causal, reps, seed, perturb=False):
    q, k, v, do = _inputs(B, H, Hkv, N, d, seed)
    o, lse = forward(q, k, v, causal=causal)
    first = backward(q, k, v, o, lse, do, causal=causal, deterministic=True)
    wsz = attn_bwd_workspace_size(batch=B, heads=H, kv_heads=Hkv, seqlen_q=N, head_dim=d, scale=1.0,
                                  deterministic=1)
    side = torch.cuda.Stream()
    for rep in range(reps):
        ws = torch.full((wsz,), 0xFF, dtype=torch.uint8, device=DEV)  # nothing may carry over
        if perturb:
            # other work on a second stream, launched just before, shifts the
            # order in which the CTAs reach each tile
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                forward(q, k, v, causal=not causal)
        again = backward(q, k, v, o, lse, do, causal=causal, deterministic=True, workspace=ws)
        torch.cuda.synchronize()
        for a, b, name in zip(first, again, ("dQ", "dK", "dV")):
            assert torch.equal(a, b), "%s differs on repeat %d" % (name, rep)
    check_device_status()
    return first, (q, k, v, o, lse, do)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_repeat_is_bitwise_identical(d, causal):
    _repeat_bitwise(2, 8, 8, 2048, d, causal, reps=3, seed=5 + d)


def test_repeat_bitwise_grouped_heads_and_concurrent_work():
    _repeat_bitwise(2, 8, 2, 1536, 128, True, reps=3, seed=77, perturb=True)


def test_dk_dv_equal_the_default_backward():
    """dK and dV are accumulated per key block in TMEM in the same step order
    by both backwards, so they agree bitwise; dQ agrees to rounding."""
    (dq, dk, dv), (q, k, v, o, lse, do) = _repeat_bitwise(2, 4, 4, 1024, 128, True, reps=1, seed=91)
    dq0, dk0, dv0 = backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(dk, dk0) and torch.equal(dv, dv0)
    assert (dq.float() - dq0.float()).abs().max().item() <= 1e-2 * dq0.float().abs().max().item()


def test_full_size_repeat_bitwise():
    """The long-head training shape (B=2, H=16, N=4096, d=128, causal): two
    runs agree bitwise."""
    q, k, v, do = qkv(2, 16, 4096, 128, 1003, device=DEV)
    o, lse = forward(q, k, v, causal=True)
    a = backward(q, k, v, o, lse, do, causal=True, deterministic=True)
    b = backward(q, k, v, o, lse, do, causal=True, deterministic=True)
    torch.cuda.synchronize()
    check_device_status()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_packed_sequences_repeat_bitwise():
    """Packed sequences (lengths 1000, 0, 513, 2048, 77; shared heads): three
    deterministic runs on 0xFF-filled workspaces agree bitwise."""
    lens = [1000, 0, 513, 2048, 77]
    T, H, Hkv, d = sum(lens), 8, 2, 128
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=DEV)
    q, do = (randn((T, H, d), 101 + i, device=DEV) for i in range(2))
    k, v = (randn((T, Hkv, d), 103 + i, device=DEV) for i in range(2))
    o, lse = forward_varlen(q, k, v, cu, max(lens), causal=True)
    first = backward_varlen(q, k, v, o, lse, do, cu, max(lens), causal=True, deterministic=True)
    wsz = attn_bwd_workspace_size(layout=FA_LAYOUT_PACKED, batch=len(lens), heads=H, kv_heads=Hkv,
                                  seqlen_q=max(lens), total_q=T, head_dim=d, scale=1.0, deterministic=1,
                                  cu_seqlens_q=cu)
    for rep in range(3):
        ws = torch.full((wsz,), 0xFF, dtype=torch.uint8, device=DEV)
        again = backward_varlen(q, k, v, o, lse, do, cu, max(lens), causal=True, deterministic=True, workspace=ws)
        torch.cuda.synchronize()
        for a, b in zip(first, again):
            assert torch.equal(a, b), "repeat %d" % rep
    check_device_status()


@pytest.mark.parametrize("causal", [False, True])
def test_bnhd_deterministic_matches_oracle_and_repeats(causal):
    """flash_attn_func's layout [B, N, H, d] with deterministic=True: parity
    with the oracle on the transposed tensors, and bitwise repeats."""
    B, N, H, Hkv, d = 2, 700, 4, 2, 128
    q, do = (randn((B, N, H, d), 111 + i, device=DEV) for i in range(2))
    k, v = (randn((B, N, Hkv, d), 113 + i, device=DEV) for i in range(2))
    o, lse = forward_bnhd(q, k, v, causal=causal)
    g1 = backward_bnhd(q, k, v, o, lse, do, causal=causal, deterministic=True)
    g2 = backward_bnhd(q, k, v, o, lse, do, causal=causal, deterministic=True)
    torch.cuda.synchronize()
    check_device_status()
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
    t = lambda x: np.ascontiguousarray(np.transpose(to64(x), (0, 2, 1, 3)))
    g = H // Hkv
    r = oracle.bwd(t(q), np.repeat(t(k), g, axis=1), np.repeat(t(v), g, axis=1), t(do), 1.0 / math.sqrt(d),
                   causal=causal)
    assert_grad(t(g1[0]), r["dq"], "dQ")
    assert_grad(t(g1[1]), r["dk"].reshape(B, Hkv, g, N, d).sum(axis=2), "dK")
    assert_grad(t(g1[2]), r["dv"].reshape(B, Hkv, g, N, d).sum(axis=2), "dV")
