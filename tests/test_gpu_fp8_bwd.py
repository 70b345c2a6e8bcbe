"""GPU parity of the FP8 backward (chapter 18 §18.6.2: the backward's
products on FP8 tensor cores, dS quantised to E5M2 for the dQ and dK
products, float32 master gradients).

The reference is the oracle's backward on the FP8 forward's dequantised
inputs Q = s_q Q8, K = s_k K8, V = s_v V8 under the dequantised upstream
gradient dO^ = s_do dO8 (the library's own E4M3 quantisation of dO, bit-exact
to the oracle's): the function whose gradients the FP8 backward computes.  On
the way the kernel rounds P to E4M3 (for dV) and dS to E5M2 (for dK and dQ),
and its D comes from the FP8 forward's bf16 O; its error is a sum of per-term
rounding errors of both signs.  The bound used, 0.1875 = 2^-3 + 2^-4 times the
oracle's max|dX| (E5M2's unit roundoff for dS plus E4M3's for the other
operand), is the reading recorded in the design notes.  Cases:
causal and not, ragged N, key lengths including 0 (exact zeros), sampled rows
at the long-sequence shape, and a bitwise repeat of dK, dV."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_10_gb300 import (backward_fp8, check_device_status, forward_fp8, quantize_fp8,
                                            quantize_fp8_qkv)
from exact_tiled_attention_10_gb300.inputs import WORKLOADS, qkv
from parity_util import _log, assert_close_abs, sample_rows, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"
FP8_GRAD_REL_TOL = 2.0 ** -3 + 2.0 ** -4


def _deq(c, s):
    return oracle.dequantize_fp8(c.cpu().numpy(), s.cpu().numpy())


def _grads(B, H, N, causal, seed, kv=None):
    q, k, v, do = qkv(B, H, N, 128, seed, device=DEV)
    (q8, sq), (k8, sk), (v8, sv) = quantize_fp8_qkv(q, k, v)
    kvd = None if kv is None else torch.tensor(kv, dtype=torch.int32, device=DEV)
    o, lse = forward_fp8(q8, k8, v8, sq, sk, sv, causal=causal, kv_lens=kvd)
    dq, dk, dv = backward_fp8(q8, k8, v8, sq, sk, sv, o, lse, do, causal=causal, kv_lens=kvd)
    torch.cuda.synchronize()
    check_device_status()
    do8, sdo = quantize_fp8(do)
    return (q8, sq, k8, sk, v8, sv, _deq(do8, sdo), kvd), (dq, dk, dv)


def _assert_fp8_grad(gpu, ref, what):
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    return assert_close_abs(gpu, ref, max(FP8_GRAD_REL_TOL * scale, 1e-5), what)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [128, 300, 777])
def test_fp8_backward_matches_oracle_on_dequantised_inputs(N, causal):
    (q8, sq, k8, sk, v8, sv, do, _), (dq, dk, dv) = _grads(2, 2, N, causal, 211 + N)
    r = oracle.bwd(_deq(q8, sq), _deq(k8, sk), _deq(v8, sv), do, 1 / math.sqrt(128), causal=causal)
    for name, x in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert x.dtype == torch.float32
        _assert_fp8_grad(to64(x), r[name], name)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_backward_against_the_original_bf16_inputs(causal):
    """Against the oracle on the ORIGINAL bf16 Q, K, V, dO (before E4M3
    quantisation), element by element: by the triangle inequality the error
    is at most the kernel's bound on the dequantised inputs plus the exact
    effect of the input quantisation, |dX(Q^, K^, V^, dO^) - dX(Q, K, V, dO)|,
    which the oracle computes on both input sets (nothing here comes from the
    GPU).  The norm-wise relative error is logged beside it."""
    N = 300
    q, k, v, do = qkv(2, 2, N, 128, 311 + causal, device=DEV)
    (q8, sq, k8, sk, v8, sv, do_hat, _), (dq, dk, dv) = _grads(2, 2, N, causal, 311 + causal)
    sc = 1 / math.sqrt(128)
    r_hat = oracle.bwd(_deq(q8, sq), _deq(k8, sk), _deq(v8, sv), do_hat, sc, causal=causal)
    r = oracle.bwd(to64(q), to64(k), to64(v), to64(do), sc, causal=causal)
    for name, x in (("dq", dq), ("dk", dk), ("dv", dv)):
        g = to64(x)
        bound = FP8_GRAD_REL_TOL * np.max(np.abs(r_hat[name])) + np.abs(r_hat[name] - r[name])
        err = np.abs(g - r[name])
        rel = np.linalg.norm(g - r[name]) / np.linalg.norm(r[name])
        _log("%s vs original inputs (norm-wise %.4f)" % (name, rel), np.max(err / np.maximum(bound, 1e-300)), 1.0,
             normwise=rel)
        assert np.all(err <= bound), "%s: %d elements over the bound" % (name, int(np.sum(err > bound)))


def test_fp8_backward_key_lengths_and_empty_items():
    kv = [0, 1, 200, 640]
    (q8, sq, k8, sk, v8, sv, do, kvd), (dq, dk, dv) = _grads(4, 2, 640, True, 223, kv=kv)
    r = oracle.bwd(_deq(q8, sq), _deq(k8, sk), _deq(v8, sv), do, 1 / math.sqrt(128), causal=True,
                   kv_lens=np.asarray(kv, dtype=np.int32))
    for name, x in (("dq", dq), ("dk", dk), ("dv", dv)):
        _assert_fp8_grad(to64(x), r[name], name)
    # batch item 0 sees no key: exact zeros; keys beyond kv_len get exactly zero dK, dV
    assert torch.all(dq[0] == 0) and torch.all(dk[0] == 0) and torch.all(dv[0] == 0)
    for b, L in enumerate(kv):
        assert torch.all(dk[b, :, L:] == 0) and torch.all(dv[b, :, L:] == 0)


def test_fp8_backward_long_sequence_sampled():
    """B=1, H=8, N=16384 (the FP8 workload's shape), non-causal: sampled rows
    and keys of two heads against the row-sampled oracle on dequantised
    inputs."""
    w = WORKLOADS["long_seq"]
    (q8, sq, k8, sk, v8, sv, do, _), (dq, dk, dv) = _grads(w.B, w.H, w.N, False, w.seed)
    rows = sample_rows(w.N, 16, seed=7)
    keys = sample_rows(w.N, 8, seed=8)
    for h in (0, 5):
        qh, kh, vh = (_deq(c[:, h:h + 1], s[:, h:h + 1])[0, 0] for c, s in ((q8, sq), (k8, sk), (v8, sv)))
        g = oracle.bwd_rows(qh, kh, vh, do[0, h], w.scale, False, w.N, rows, keys)
        _assert_fp8_grad(to64(dq[0, h])[rows], g["dq"], "dQ rows")
        _assert_fp8_grad(to64(dk[0, h])[keys], g["dk"], "dK keys")
        _assert_fp8_grad(to64(dv[0, h])[keys], g["dv"], "dV keys")


def test_fp8_backward_repeat_is_bitwise_for_dk_dv():
    """dK, dV of every key block come from one CTA in a fixed order: repeats
    agree bit for bit (dQ is summed by float32 reductions in varying order)."""
    q, k, v, do = qkv(2, 4, 1000, 128, 229, device=DEV)
    (q8, sq), (k8, sk), (v8, sv) = quantize_fp8_qkv(q, k, v)
    o, lse = forward_fp8(q8, k8, v8, sq, sk, sv, causal=True)
    dq, dk, dv = backward_fp8(q8, k8, v8, sq, sk, sv, o, lse, do, causal=True)
    for _ in range(2):
        dq2, dk2, dv2 = backward_fp8(q8, k8, v8, sq, sk, sv, o, lse, do, causal=True)
        torch.cuda.synchronize()
        assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
        assert (dq - dq2).abs().max().item() <= 1e-3 * dq.abs().max().item()
    check_device_status()
