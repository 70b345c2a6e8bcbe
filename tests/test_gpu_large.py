"""The largest sizes: tensors of more than 2^31 elements (B = 1, H = 1025,
N = 16384, d = 128; 2.15e9 elements, 4.3 GB each in bf16), so that every
element offset past the first 2^31 needs 64-bit index arithmetic in the
kernels.  Causal forward and backward; the LAST head, whose elements all lie
beyond 2^31, is checked against the oracle on sampled rows and keys (O, LSE,
dQ rows; dK, dV keys), and the whole output against properties that hold at
any size: every value finite, and per head the column sums of dV equal those
of dO (each query row's probabilities sum to 1), and <dQ, Q> = <dK, K> (both
are scale * sum_ij dS_ij q_i.k_j)."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_10_gb300 import backward, check_device_status, forward
from exact_tiled_attention_10_gb300.inputs import randn_on_device
from parity_util import assert_grad, assert_lse, assert_o, sample_rows, to64

pytestmark = pytest.mark.gpu


def test_more_than_2_31_elements_causal():
    B, H, N, d = 1, 1025, 16384, 128
    assert B * H * N * d > 2 ** 31
    free, _ = torch.cuda.mem_get_info()
    if free < 60 * 2 ** 30:
        pytest.skip("needs ~45 GB of free device memory")
    shape = (B, H, N, d)
    q, k, v, do = (randn_on_device(shape, 4100 + i, "cuda") for i in range(4))
    scale = 1.0 / math.sqrt(d)
    o, lse = forward(q, k, v, causal=True)
    dq, dk, dv = backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    check_device_status()
    h = H - 1
    rows = sample_rows(N, 16, seed=11)
    keys = sample_rows(N, 8, seed=12)
    qh, kh, vh, gh = (to64(t[0, h]) for t in (q, k, v, do))
    ro, rl = oracle.fwd_rows(qh, kh, vh, scale, True, N, rows)
    assert_o(to64(o[0, h])[rows], ro, "O rows, last head")
    assert_lse(to64(lse[0, h])[rows], rl, what="LSE rows, last head")
    g = oracle.bwd_rows(qh, kh, vh, gh, scale, True, N, rows, keys)
    assert_grad(to64(dq[0, h])[rows], g["dq"], "dQ rows, last head")
    assert_grad(to64(dk[0, h])[keys], g["dk"], "dK keys, last head")
    assert_grad(to64(dv[0, h])[keys], g["dv"], "dV keys, last head")
    # properties over every head (float64 sums of the device tensors)
    for t in (o, lse, dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    f64 = lambda t: t.double()
    for h0 in range(0, H, 64):
        sl = slice(h0, min(H, h0 + 64))
        cs_dv = f64(dv[0, sl]).sum(1)  # [heads, d]
        cs_do = f64(do[0, sl]).sum(1)
        assert torch.allclose(cs_dv, cs_do, rtol=0, atol=5e-3 * cs_do.abs().max().item())
        ip_q = (f64(dq[0, sl]) * f64(q[0, sl])).sum((1, 2))
        ip_k = (f64(dk[0, sl]) * f64(k[0, sl])).sum((1, 2))
        norm = lambda a, b: f64(a[0, sl]).norm(dim=(1, 2)) * f64(b[0, sl]).norm(dim=(1, 2))
        tol = 1e-2 * (norm(dq, q) + norm(dk, k))
        assert bool(((ip_q - ip_k).abs() <= tol).all())
