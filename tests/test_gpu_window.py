"""GPU parity of sliding-window attention (chapter 18 §18.7.1, window_size =
(left, right): key j visible to query i only if i - left <= j <= i + right,
-1 = unbounded; §18.8.1: key blocks outside every row's window are skipped).

The oracle applies the window mask element by element on the materialised
S; the GPU skips whole blocks outside a tile's window and masks the boundary
blocks.  Cases cover windows narrower than, equal to and wider than a tile,
one-sided windows, window (0, 0), the window combined with the causal and
key-padding masks, shared key/value heads, sequence lengths off the tile
grid, and a long sequence checked on sampled rows and keys.  O is held to
the flat 1e-2 except on rows that see fewer than 16 keys (narrow windows),
which are held to the worst case of the kernel's two bf16 roundings
(parity_util.assert_o); LSE and the gradients keep their tolerances."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_10_gb300 import backward, check_device_status, forward
from exact_tiled_attention_10_gb300.inputs import qkv
from parity_util import assert_close_abs, assert_grad, assert_lse, assert_o, rounding_context, sample_rows, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(B, H, Hkv, N, d, causal, window, kv=None, seed=5, deterministic=False):
    q, _, _, do = qkv(B, H, N, d, seed, device=DEV)
    _, k, v = qkv(B, Hkv, N, d, seed + 50, device=DEV, with_dout=False)
    kvd = None if kv is None else torch.tensor(kv, dtype=torch.int32, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = forward(q, k, v, causal=causal, scale=scale, kv_lens=kvd, window=window)
    dq, dk, dv = backward(q, k, v, o, lse, do, causal=causal, scale=scale, kv_lens=kvd, window=window,
                          deterministic=deterministic)
    torch.cuda.synchronize()
    check_device_status()
    if deterministic:  # a second run agrees bit for bit
        again = backward(q, k, v, o, lse, do, causal=causal, scale=scale, kv_lens=kvd, window=window,
                         deterministic=True)
        torch.cuda.synchronize()
        for a, b in zip((dq, dk, dv), again):
            assert torch.equal(a, b)
    g = H // Hkv
    kvn = None if kv is None else np.asarray(kv, dtype=np.int32)
    kr, vr = np.repeat(to64(k), g, axis=1), np.repeat(to64(v), g, axis=1)
    ref = oracle.bwd(to64(q), kr, vr, to64(do), scale, causal=causal, kv_lens=kvn, window=window)
    nvis, absref = rounding_context(
        lambda qq, vv: oracle.fwd(qq, kr, vv, scale, causal=causal, kv_lens=kvn, window=window), to64(q), vr)
    assert_o(to64(o), ref["o"], nvis=nvis, absref=absref)
    assert_lse(to64(lse), ref["lse"])
    assert_grad(to64(dq), ref["dq"], "dQ")
    assert_grad(to64(dk), ref["dk"].reshape(B, Hkv, g, N, d).sum(axis=2), "dK")
    assert_grad(to64(dv), ref["dv"].reshape(B, Hkv, g, N, d).sum(axis=2), "dV")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal,window", [
    (True, (64, -1)), (True, (200, 0)), (False, (100, 37)), (False, (0, 0)), (False, (-1, 50)),
    (False, (255, -1)), (False, (130, 130)), (True, (1000, 1000)),
])
def test_window_matches_oracle(d, causal, window):
    _case(2, 2, 2, 600, d, causal, window, seed=7 + d + window[0])


def test_window_with_key_padding_and_shared_heads():
    _case(3, 4, 2, 389, 128, False, (90, 20), kv=[0, 150, 389], seed=31)
    _case(2, 4, 1, 300, 64, True, (40, -1), kv=[1, 257], seed=37)


def test_window_wider_than_sequence_equals_plain_forward():
    q, k, v = qkv(1, 4, 520, 128, 41, device=DEV, with_dout=False)
    for causal in (False, True):
        o1, l1 = forward(q, k, v, causal=causal)
        o2, l2 = forward(q, k, v, causal=causal, window=(520, 520))
        torch.cuda.synchronize()
        assert_close_abs(to64(o2), to64(o1), 2e-3, "O (wide window vs none)")
        assert_lse(to64(l2), to64(l1), 1e-4)


def test_window_long_sequence_sampled():
    """N = 8192, d = 128, a causal window of 1024 (the Mistral-style pattern):
    sampled query rows and keys of two heads against the row-sampled oracle."""
    B, H, N, d = 1, 4, 8192, 128
    window = (1024, -1)
    q, k, v, do = qkv(B, H, N, d, 43, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = forward(q, k, v, causal=True, scale=scale, window=window)
    dq, dk, dv = backward(q, k, v, o, lse, do, causal=True, scale=scale, window=window)
    torch.cuda.synchronize()
    check_device_status()
    rows = sample_rows(N, 24, seed=3) + [1023, 1024, 1025, 4100]
    rows = sorted(set(rows))
    keys = sorted(set(sample_rows(N, 12, seed=4)))
    for h in (0, 3):
        qh, kh, vh, gh = (to64(t[0, h]) for t in (q, k, v, do))
        run = lambda qq, vv: oracle.fwd_rows(qq, kh, vv, scale, True, N, rows, window=window)
        o_ref, lse_ref = run(qh, vh)
        nvis, absref = rounding_context(run, qh, vh)
        assert_o(to64(o[0, h])[rows], o_ref, "O rows", nvis=nvis, absref=absref)
        assert_lse(to64(lse[0, h])[rows], lse_ref)
        # gradient scale: the oracle's max-abs over the sampled rows / keys
        g = oracle.bwd_rows(qh, kh, vh, gh, scale, True, N, rows, keys, window=window)
        assert_grad(to64(dq[0, h])[rows], g["dq"], "dQ rows")
        assert_grad(to64(dk[0, h])[keys], g["dk"], "dK keys")
        assert_grad(to64(dv[0, h])[keys], g["dv"], "dV keys")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal,window", [(True, (200, 0)), (False, (100, 37)), (False, (-1, 50)),
                                           (False, (130, 130)), (True, (64, -1))])
def test_window_deterministic(d, causal, window):
    """The deterministic backward under a sliding window: the key blocks that
    visit a query block start above 0, and each takes its rank within that
    range; parity with the oracle and a bitwise repeat."""
    _case(2, 4, 2, 1100, d, causal, window, kv=[1100, 777], seed=91 + d + window[0], deterministic=True)
