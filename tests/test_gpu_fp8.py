"""GPU parity of the FP8 E4M3 path (chapter 18 §18.6.2): the per-block
quantiser must reproduce the oracle's codes and scales exactly (a byte-level
result decided in float32 on both sides); the FP8 forward must match the
oracle within 6e-2 max-abs on O.

The FP8 workload of the pages is non-causal; there the reference is the oracle
on the ORIGINAL bf16 inputs.  With a causal mask the first rows average only a
handful of value rows, so the E4M3 rounding of V itself (up to 2^-4 relative)
is not averaged away; causal cases are therefore checked against the oracle on
the dequantised inputs s * X8, which isolates the kernel's own arithmetic."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_10_gb300 import check_device_status, forward_fp8, quantize_fp8, quantize_fp8_qkv
from exact_tiled_attention_10_gb300.inputs import WORKLOADS, kv_lens_ragged, qkv, randn
from parity_util import FP8_O_TOL, assert_close_abs, assert_lse, sample_rows, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("N", [1, 63, 64, 65, 300, 1024])
@pytest.mark.parametrize("d", [64, 128])
def test_quantiser_bit_exact(N, d):
    x = qkv(2, 3, N, d, 40 + N, device=DEV, with_dout=False)[0]
    x[0, 0, : min(N, 64)] = 0  # an all-zero block takes scale 1
    c, s = quantize_fp8(x)
    torch.cuda.synchronize()
    rc, rs = oracle.quantize_fp8(x)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    np.testing.assert_array_equal(c.cpu().numpy(), rc)


def test_quantiser_bit_exact_long_seq_head():
    w = WORKLOADS["long_seq"]
    q = qkv(w.B, w.H, w.N, w.d, w.seed, device=DEV, with_dout=False)[0]
    c, s = quantize_fp8(q)
    torch.cuda.synchronize()
    sub = q[:, :2].contiguous()  # two whole heads through the oracle
    rc, rs = oracle.quantize_fp8(sub)
    np.testing.assert_array_equal(s[:, :2].cpu().numpy(), rs)
    np.testing.assert_array_equal(c[:, :2].cpu().numpy(), rc)


def test_quantiser_division_matches_ieee_bitwise():
    """The quantiser divides by a scale shared by a whole block with one
    reciprocal and a fused-multiply-add correction (Markstein's method); its
    quotients must equal IEEE float32 division bit for bit, or the E4M3 codes
    could differ from the oracle's at rounding midpoints."""
    import ctypes
    from exact_tiled_attention_10_gb300 import load_library
    g = torch.Generator(device="cpu").manual_seed(77)
    n, ns = 1 << 24, 4096
    x = (torch.randn(n, generator=g) * torch.exp2(torch.randint(-20, 21, (n,), generator=g).float()))
    x = x.to(torch.bfloat16).float()  # the quantiser's dividends are bf16 values
    amax = torch.rand(ns, generator=g) * torch.exp2(torch.randint(-60, 61, (ns,), generator=g).float())
    s = (amax.to(torch.bfloat16).float() / 448.0).clamp_min(1e-30)
    s[:64] = torch.exp2(torch.arange(-32, 32).float())  # exact powers of two
    x, s = x.to(DEV), s.to(DEV)
    qf, qi = torch.empty_like(x), torch.empty_like(x)
    lib = load_library()
    st = lib.fa_selftest_quantiser_division(x.data_ptr(), s.data_ptr(), ns, n, qf.data_ptr(), qi.data_ptr(),
                                            torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    bad = (qf.view(torch.int32) != qi.view(torch.int32)).sum().item()
    assert bad == 0, "%d quotients differ from IEEE division" % bad


@pytest.mark.parametrize("mag", [1e35, 1e-35, 1e-3, 1e3])
def test_quantiser_bit_exact_extreme_scales(mag):
    """Scales outside the shared-divisor range take IEEE division; both paths
    must still reproduce the oracle's codes."""
    x = (qkv(1, 2, 200, 128, 91, device=DEV, with_dout=False)[0].float() * mag).to(torch.bfloat16)
    c, s = quantize_fp8(x)
    torch.cuda.synchronize()
    rc, rs = oracle.quantize_fp8(x)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    np.testing.assert_array_equal(c.cpu().numpy(), rc)


def test_quantise_qkv_in_one_launch_equals_separate_calls():
    from exact_tiled_attention_10_gb300 import quantize_fp8_qkv
    q = qkv(2, 4, 333, 128, 95, device=DEV, with_dout=False)[0]
    _, k, v = qkv(2, 2, 333, 128, 96, device=DEV, with_dout=False)
    fused = quantize_fp8_qkv(q, k, v)
    torch.cuda.synchronize()
    for (c, s), x in zip(fused, (q, k, v)):
        c1, s1 = quantize_fp8(x)
        torch.cuda.synchronize()
        assert torch.equal(c, c1) and torch.equal(s, s1)


def _fp8_run(B, H, N, seed, causal, kv=None):
    q, k, v = qkv(B, H, N, 128, seed, device=DEV, with_dout=False)
    (q8, sq), (k8, sk), (v8, sv) = (quantize_fp8(t) for t in (q, k, v))
    kvd = None if kv is None else torch.tensor(kv, dtype=torch.int32, device=DEV)
    o, lse = forward_fp8(q8, k8, v8, sq, sk, sv, causal=causal, kv_lens=kvd)
    torch.cuda.synchronize()
    check_device_status()
    return (q, k, v), (q8, sq, k8, sk, v8, sv), o, lse


@pytest.mark.parametrize("N", [1024, 2048])
def test_fp8_forward_noncausal_vs_bf16_inputs(N):
    (q, k, v), _, o, lse = _fp8_run(2, 2, N, 70 + N, False)
    ref_o, ref_l = oracle.fwd(to64(q), to64(k), to64(v), 1 / math.sqrt(128))
    assert_close_abs(to64(o), ref_o, FP8_O_TOL, "FP8 O")


def p_rounding_bound(q, k, v, o_ref, lse_ref, causal, kv):
    """Largest |O - O_ref| that rounding each probability weight to E4M3
    (relative error <= 2^-4 in the normal range, the normaliser summing the
    rounded weights) can cause, per element: 2^-4/(1-2^-4) * sum_j P_ij
    |v_j - O_i|, plus the bf16 rounding of the output (2^-8 |O_i|) and 1e-3
    for subnormal weights and float32 accumulation.  P is evaluated from the oracle's LSE; it sets a
    tolerance only, never an expected value."""
    B, H, N, d = q.shape
    scale = 1 / math.sqrt(d)
    out = np.zeros_like(o_ref)
    for b in range(B):
        for h in range(H):
            S = scale * q[b, h] @ k[b, h].T
            vis = np.arange(N)[None, :] < kv[b]
            if causal:
                vis = vis & (np.arange(N)[None, :] <= np.arange(N)[:, None])
            L = lse_ref[b, h][:, None]
            P = np.where(vis & np.isfinite(L), np.exp(np.where(vis, S, 0.0) - np.where(np.isfinite(L), L, 0.0)), 0.0)
            dev = np.abs(v[b, h][None, :, :] - o_ref[b, h][:, None, :])  # [N, N, d]
            out[b, h] = np.einsum("ij,ijt->it", P, dev)
    return out * (2.0 ** -4 / (1 - 2.0 ** -4)) + 2.0 ** -8 * np.abs(o_ref) + 1e-3


@pytest.mark.parametrize("N", [100, 300, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_vs_dequantised_inputs(N, causal):
    kv = [N, N // 3 + 1]
    _, (q8, sq, k8, sk, v8, sv), o, lse = _fp8_run(2, 2, N, 90 + N, causal, kv=kv)
    dq = oracle.dequantize_fp8(q8.cpu().numpy(), sq.cpu().numpy())
    dk = oracle.dequantize_fp8(k8.cpu().numpy(), sk.cpu().numpy())
    dv = oracle.dequantize_fp8(v8.cpu().numpy(), sv.cpu().numpy())
    ref_o, ref_l = oracle.fwd(dq, dk, dv, 1 / math.sqrt(128), causal=causal,
                              kv_lens=np.array(kv, dtype=np.int32))
    # O: the 6e-2 target, and per element the bound that E4M3 rounding of the
    # probabilities allows (see p_rounding_bound)
    og = to64(o)
    if not causal:
        assert_close_abs(og, ref_o, FP8_O_TOL, "FP8 O (dequantised reference)")
    bound = p_rounding_bound(dq, dk, dv, ref_o, ref_l, causal, kv)
    excess = np.abs(og - ref_o) - bound
    assert np.all(excess <= 0), "FP8 O exceeds the E4M3 probability-rounding bound by %.3e" % excess.max()
    # LSE uses exact float32 scores of the quantised operands and the exact sum
    assert_lse(to64(lse), ref_l, what="FP8 LSE (dequantised reference)")


def test_fp8_long_seq_config_sampled():
    """The FP8 workload: B=1, H=8, N=16384, d=128, non-causal, per-64x128-block
    scales, bf16 output; sampled rows of two heads against the oracle on the
    original bf16 inputs."""
    w = WORKLOADS["long_seq"]
    (q, k, v), _, o, lse = _fp8_run(w.B, w.H, w.N, w.seed, False)
    assert torch.isfinite(o.float()).all()
    for h in (0, 7):
        rows = sample_rows(w.N, 40, seed=h)
        ref_o, ref_l = oracle.fwd_rows(to64(q[0, h]), to64(k[0, h]), to64(v[0, h]), w.scale, False,
                                       w.N, rows)
        assert_close_abs(to64(o[0, h, rows]), ref_o, FP8_O_TOL, "FP8 O[0,%d]" % h)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hkv", [1, 2])
def test_fp8_forward_shared_kv_heads(causal, Hkv):
    """FP8 forward with fewer key/value heads (quantised together with
    fa_quantize_fp8_qkv): bitwise the same O and LSE as the FP8 forward on
    explicitly repeated codes and scales, and, against the oracle on the
    dequantised inputs (key/value heads broadcast), O within the E4M3
    probability-rounding bound and LSE within its tolerance."""
    B, H, N = 2, 4, 300
    kv = [N, 117]
    q = randn((B, H, N, 128), 151, device=DEV)
    k = randn((B, Hkv, N, 128), 152, device=DEV)
    v = randn((B, Hkv, N, 128), 153, device=DEV)
    (q8, sq), (k8, sk), (v8, sv) = quantize_fp8_qkv(q, k, v)
    kvd = torch.tensor(kv, dtype=torch.int32, device=DEV)
    o, lse = forward_fp8(q8, k8, v8, sq, sk, sv, causal=causal, kv_lens=kvd)
    g = H // Hkv
    rep = lambda t: t.repeat_interleave(g, dim=1).contiguous()
    o_rep, lse_rep = forward_fp8(q8, rep(k8), rep(v8), sq, rep(sk), rep(sv), causal=causal, kv_lens=kvd)
    torch.cuda.synchronize()
    check_device_status()
    assert torch.equal(o, o_rep) and torch.equal(lse, lse_rep)
    dq = oracle.dequantize_fp8(q8.cpu().numpy(), sq.cpu().numpy())
    dk = np.repeat(oracle.dequantize_fp8(k8.cpu().numpy(), sk.cpu().numpy()), g, axis=1)
    dv = np.repeat(oracle.dequantize_fp8(v8.cpu().numpy(), sv.cpu().numpy()), g, axis=1)
    ref_o, ref_l = oracle.fwd(dq, dk, dv, 1 / math.sqrt(128), causal=causal, kv_lens=np.array(kv, dtype=np.int32))
    bound = p_rounding_bound(dq, dk, dv, ref_o, ref_l, causal, kv)
    excess = np.abs(to64(o) - ref_o) - bound
    assert np.all(excess <= 0), "FP8 O exceeds the E4M3 probability-rounding bound by %.3e" % excess.max()
    assert_lse(to64(lse), ref_l, what="FP8 LSE (dequantised reference)")
