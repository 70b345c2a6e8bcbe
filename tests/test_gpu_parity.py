"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, element
by element on small shapes that span several tiles and ragged tails, and on
sampled rows at the full workload sizes in the launch configuration the
benchmark times."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_10_gb300 import backward, check_device_status, forward
from exact_tiled_attention_10_gb300.inputs import WORKLOADS, kv_lens_ragged, qkv
from parity_util import assert_grad, assert_lse, assert_o, sample_rows, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run_full(B, H, N, d, causal, kv=None, dtype=torch.bfloat16, seed=7, block_c=0, do_bwd=True):
    q, k, v, do = qkv(B, H, N, d, seed, dtype=dtype, device=DEV)
    kvd = None if kv is None else torch.tensor(kv, dtype=torch.int32, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = forward(q, k, v, causal=causal, scale=scale, kv_lens=kvd, block_c=block_c)
    if do_bwd:
        dq, dk, dv = backward(q, k, v, o, lse, do, causal=causal, scale=scale, kv_lens=kvd)
    torch.cuda.synchronize()
    check_device_status()
    kvn = None if kv is None else np.asarray(kv, dtype=np.int32)
    ref = oracle.bwd(to64(q), to64(k), to64(v), to64(do), scale, causal=causal, kv_lens=kvn)
    assert_o(to64(o), ref["o"])
    assert_lse(to64(lse), ref["lse"])
    if do_bwd:
        assert_grad(to64(dq), ref["dq"], "dQ")
        assert_grad(to64(dk), ref["dk"], "dK")
        assert_grad(to64(dv), ref["dv"], "dV")
    return ref


# ----------------------------------------------------------------- tiny config
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block_c", [64, 128])
def test_tiny_config(dtype, causal, block_c):
    w = WORKLOADS["tiny"]
    _run_full(w.B, w.H, w.N, w.d, causal, dtype=dtype, seed=w.seed, block_c=block_c)


# ------------------------------------------------------ ragged tails, many tiles
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 17, 100, 129, 200, 257, 383, 520])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(d, N, causal):
    _run_full(2, 2, N, d, causal, seed=100 + N)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_key_padding(d, causal):
    N = 300
    kv = [0, 1, 63, 64, 65, 128, 129, 300]
    _run_full(len(kv), 2, N, d, causal, kv=kv, seed=31)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("block_c", [64, 128])
def test_block_sizes_agree(d, block_c):
    _run_full(1, 3, 640, d, True, seed=5, block_c=block_c, do_bwd=False)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_row_max_jumps_in_later_blocks(d, causal):
    """Running-state updates when a later key block holds a far larger score
    (FA-v2 analysis page §2.3: O is rescaled by exp(m_old - m_new) whenever the
    maximum moves).  Every query gets a common direction u, key 300 (block 2)
    scores about 25 above the rest in log2 units and key 600 (block 4) about 95,
    so both the moderate move of the reference maximum and the large one are
    exercised, for some rows of a warp and not others under the causal mask.
    Only the forward is compared: with one key holding all the weight the
    gradients nearly vanish (dS = P (dP - D) cancels), so an element-wise bound
    relative to their tiny maximum would measure float32 cancellation only."""
    B, H, N = 1, 2, 700
    q, k, v = qkv(B, H, N, d, 404 + d, device=DEV, with_dout=False)
    u = torch.ones(d, dtype=torch.float32, device=DEV) / math.sqrt(d)
    gain = math.sqrt(d) / (5.0 * math.log2(math.e))  # key amplitude per log2 unit of score
    qf = q.float() + 5.0 * u
    kf = k.float()
    kf[:, :, 300] = 25.0 * gain * u
    kf[:, :, 600] = 95.0 * gain * u
    q, k = qf.to(torch.bfloat16), kf.to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    o, lse = forward(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    check_device_status()
    o_ref, lse_ref = oracle.fwd(to64(q), to64(k), to64(v), scale, causal=causal)
    assert_o(to64(o), o_ref)
    assert_lse(to64(lse), lse_ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_repeat_is_bitwise_consistent(d, causal):
    """Race check: every key block's dK, dV is produced by one CTA in a fixed
    order, so repeated runs must agree bitwise (dQ is summed by float32
    reductions whose order varies, so it agrees to rounding); the forward is
    bitwise deterministic."""
    q, k, v, do = qkv(2, 8, 2048, d, 3, device=DEV)
    o, lse = forward(q, k, v, causal=causal)
    g1 = backward(q, k, v, o, lse, do, causal=causal)
    for _ in range(3):
        g2 = backward(q, k, v, o, lse, do, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
        assert (g1[0].float() - g2[0].float()).abs().max().item() <= 1e-2 * g1[0].float().abs().max().item()
        o2, lse2 = forward(q, k, v, causal=causal)
        assert torch.equal(o, o2) and torch.equal(lse, lse2)
    check_device_status()


# ------------------------------------------------- full workload sizes
def _full_check(w, causal, kv=None):
    """Every element of O, LSE, dQ, dK, dV of the whole workload against the
    oracle (fp64, one thread per head)."""
    q, k, v, do = qkv(w.B, w.H, w.N, w.d, w.seed, device=DEV)
    o, lse = forward(q, k, v, causal=causal, kv_lens=kv)
    dq, dk, dv = backward(q, k, v, o, lse, do, causal=causal, kv_lens=kv)
    torch.cuda.synchronize()
    check_device_status()
    kvn = None if kv is None else kv.cpu().numpy()
    ref = oracle.bwd(to64(q), to64(k), to64(v), to64(do), w.scale, causal=causal, kv_lens=kvn)
    assert_o(to64(o), ref["o"])
    assert_lse(to64(lse), ref["lse"])
    assert_grad(to64(dq), ref["dq"], "dQ")
    assert_grad(to64(dk), ref["dk"], "dK")
    assert_grad(to64(dv), ref["dv"], "dV")
    return q, k, v, do, o, lse, (dq, dk, dv)


def _sampled_check(w, causal, heads, n_rows=48, bwd=True, seed_off=0):
    """Sampled rows and keys of some heads at a size whose full oracle does not
    finish in seconds.  The gradient scale is the oracle's max-abs over the
    sampled rows / keys (a lower bound of the whole tensor's, so the check is
    at least as strict as a full one); nothing is scaled by the GPU's output."""
    q, k, v, do = qkv(w.B, w.H, w.N, w.d, w.seed, device=DEV)
    kv = kv_lens_ragged(w.B, w.N, w.seed, device=DEV) if w.ragged else None
    o, lse = forward(q, k, v, causal=causal, kv_lens=kv)
    if bwd:
        dq, dk, dv = backward(q, k, v, o, lse, do, causal=causal, kv_lens=kv)
    torch.cuda.synchronize()
    check_device_status()
    assert torch.isfinite(o.float()).all()
    kvn = None if kv is None else kv.cpu().numpy()
    for (b, h) in heads:
        kvl = w.N if kvn is None else int(kvn[b])
        rows = sample_rows(w.N, n_rows, seed=b * 131 + h + seed_off)
        qh, kh, vh = to64(q[b, h]), to64(k[b, h]), to64(v[b, h])
        o_ref, lse_ref = oracle.fwd_rows(qh, kh, vh, w.scale, causal, kvl, rows)
        assert_o(to64(o[b, h, rows]), o_ref, "O[%d,%d]" % (b, h))
        assert_lse(to64(lse[b, h, rows]), lse_ref, what="LSE[%d,%d]" % (b, h))
        if bwd:
            keys = sample_rows(w.N, n_rows // 2, seed=b * 7 + h + 1 + seed_off)
            g = oracle.bwd_rows(qh, kh, vh, to64(do[b, h]), w.scale, causal, kvl, rows, keys)
            for name, x, ref, idx in (("dQ", dq, g["dq"], rows), ("dK", dk, g["dk"], keys),
                                      ("dV", dv, g["dv"], keys)):
                assert_grad(to64(x[b, h, idx]), ref, "%s[%d,%d]" % (name, b, h))
    return q, k, v, o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_mid_config_full(causal):
    """B=4, H=16, N=2048, d=64: the whole workload, element by element."""
    _full_check(WORKLOADS["mid"], causal)


def test_long_head_config_full_heads():
    """B=2, H=16, N=4096, d=128, causal (the benchmark's launch): two whole heads
    element by element (the oracle on all 64 heads would take minutes), the
    rest of the tensors finite."""
    w = WORKLOADS["long_head"]
    q, k, v, do = qkv(w.B, w.H, w.N, w.d, w.seed, device=DEV)
    o, lse = forward(q, k, v, causal=True)
    dq, dk, dv = backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    check_device_status()
    for t in (o, dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    heads = [(0, 0), (1, 15)]
    pick = lambda t: np.stack([to64(t[b, h]) for b, h in heads])[None]
    ref = oracle.bwd(pick(q), pick(k), pick(v), pick(do), w.scale, causal=True)
    assert_o(pick(o), ref["o"])
    assert_lse(np.stack([to64(lse[b, h]) for b, h in heads])[None], ref["lse"])
    assert_grad(pick(dq), ref["dq"], "dQ")
    assert_grad(pick(dk), ref["dk"], "dK")
    assert_grad(pick(dv), ref["dv"], "dV")


def test_long_head_noncausal_forward_sampled():
    w = WORKLOADS["long_head"]
    _sampled_check(w, False, heads=[(1, 3)], bwd=False, seed_off=5)


def test_ragged_config_full():
    """B=8, H=32, N=1024, d=128 with per-item key lengths (item 0: none): the
    whole workload element by element, and the exact zeros the fully-masked
    convention fixes (attention-kernels wiki §04)."""
    w = WORKLOADS["ragged"]
    kv = kv_lens_ragged(w.B, w.N, w.seed, device=DEV)
    assert int(kv[0]) == 0
    q, k, v, do, o, lse, (dq, dk, dv) = _full_check(w, False, kv=kv)
    # batch item 0 has kv_len = 0: every row fully masked -> O = 0, LSE = -inf, zero grads
    assert torch.all(o[0] == 0)
    assert torch.all(torch.isneginf(lse[0]))
    assert torch.all(dq[0] == 0) and torch.all(dk[0] == 0) and torch.all(dv[0] == 0)
    # keys beyond kv_len get exactly zero dK, dV
    for b in range(1, w.B):
        L = int(kv[b])
        assert torch.all(dk[b, :, L:] == 0) and torch.all(dv[b, :, L:] == 0)


def test_long_seq_config_sampled():
    w = WORKLOADS["long_seq"]
    _sampled_check(w, True, heads=[(0, 0), (0, 5)], n_rows=32)
