"""GPU parity of packed variable-length sequences (chapter 18 §18.7.1,
flash_attn_varlen_func: sequences of unequal length concatenated token by
token, offsets in cu_seqlens, no attention across sequence boundaries, the
causal mask applied within each sequence).  The reference runs the oracle on
each sequence alone (its tokens as one [1, H, len, d] problem, key/value
heads broadcast for grouped heads) and compares every token of O, LSE, dQ,
dK, dV; sequences of length 0 and 1 and lengths off the 64/128 tile grid
are included."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_10_gb300 import backward_varlen, check_device_status, forward_varlen
from exact_tiled_attention_10_gb300.inputs import randn
from parity_util import FEW_KEYS, assert_grad, assert_lse, assert_o, rounding_context, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(lens, H, Hkv, d, causal, seed, deterministic=False, window=None):
    T = int(sum(lens))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=DEV)
    q = randn((T, H, d), seed, device=DEV)
    k = randn((T, Hkv, d), seed + 1, device=DEV)
    v = randn((T, Hkv, d), seed + 2, device=DEV)
    do = randn((T, H, d), seed + 3, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = forward_varlen(q, k, v, cu, max(lens), causal=causal, scale=scale, window=window)
    dq, dk, dv = backward_varlen(q, k, v, o, lse, do, cu, max(lens), causal=causal, scale=scale,
                                 deterministic=deterministic, window=window)
    torch.cuda.synchronize()
    check_device_status()
    if deterministic:  # a second run agrees bit for bit
        again = backward_varlen(q, k, v, o, lse, do, cu, max(lens), causal=causal, scale=scale,
                                deterministic=True, window=window)
        torch.cuda.synchronize()
        for a, b in zip((dq, dk, dv), again):
            assert torch.equal(a, b)
    g = H // Hkv
    # reference, one sequence at a time
    ref = {n: np.zeros(t.shape) for n, t in (("o", q), ("dq", q), ("dk", k), ("dv", v))}
    ref_lse = np.zeros((H, T))
    nvis = np.full((T, H), FEW_KEYS, dtype=np.float64)
    absref = np.zeros((T, H, d))
    a = 0
    for n in lens:
        if n > 0:
            sl = slice(a, a + n)
            per = lambda t, rep: np.repeat(to64(t[sl]).transpose(1, 0, 2)[None], rep, axis=1)
            r = oracle.bwd(per(q, 1), per(k, g), per(v, g), per(do, 1), scale, causal=causal, window=window)
            ref["o"][sl] = r["o"][0].transpose(1, 0, 2)
            ref["dq"][sl] = r["dq"][0].transpose(1, 0, 2)
            ref["dk"][sl] = r["dk"][0].reshape(Hkv, g, n, d).sum(axis=1).transpose(1, 0, 2)
            ref["dv"][sl] = r["dv"][0].reshape(Hkv, g, n, d).sum(axis=1).transpose(1, 0, 2)
            ref_lse[:, sl] = r["lse"][0]
            if window is not None:
                kr = per(k, g)
                nv, ab = rounding_context(lambda qq, vv: oracle.fwd(qq, kr, vv, scale, causal=causal, window=window),
                                          per(q, 1), per(v, g))
                nvis[sl] = nv[0].T
                absref[sl] = ab[0].transpose(1, 0, 2)
        a += n
    if window is None:
        assert_o(to64(o), ref["o"])
    else:  # narrow windows: rows with few keys take the rounding bound (see the window tests)
        assert_o(to64(o), ref["o"], nvis=nvis, absref=absref)
    assert_lse(to64(lse), ref_lse)
    assert_grad(to64(dq), ref["dq"], "dQ")
    assert_grad(to64(dk), ref["dk"], "dK")
    assert_grad(to64(dv), ref["dv"], "dV")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal,window", [(True, (100, 0)), (False, (64, 37)), (False, (-1, 20)), (True, (300, -1))])
def test_varlen_sliding_window(d, causal, window):
    """flash_attn_varlen_func's window_size: the window within each sequence."""
    _case([300, 1, 0, 129, 520, 64], 4, 2, d, causal, seed=151 + d + window[0], window=window)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_per_sequence_oracle(d, causal):
    _case([300, 1, 0, 129, 520, 64], 4, 4, d, causal, seed=61 + d)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_with_shared_kv_heads(causal):
    _case([200, 385, 17], 6, 2, 128, causal, seed=73)


def test_varlen_single_sequence():
    _case([777], 2, 1, 64, True, seed=79)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_deterministic_matches_oracle(d, causal):
    """The deterministic backward of packed sequences (flash_attn_varlen_func's
    deterministic flag) against the same per-sequence oracle."""
    _case([300, 1, 0, 129, 520, 64], 4, 2, d, causal, seed=91 + d, deterministic=True)


def _case_kv(lens_q, lens_k, H, Hkv, d, causal, seed, deterministic=False):
    """Separate query and key ranges (flash_attn_varlen_func's cu_seqlens_q /
    cu_seqlens_k): each sequence against the oracle's rectangular forward and
    backward (chapter 18 §18.8.2 reading: the queries are the last len_q
    positions under the causal mask)."""
    Tq, Tk = int(sum(lens_q)), int(sum(lens_k))
    cuq = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32, device=DEV)
    cuk = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32, device=DEV)
    q = randn((Tq, H, d), seed, device=DEV)
    k = randn((Tk, Hkv, d), seed + 1, device=DEV)
    v = randn((Tk, Hkv, d), seed + 2, device=DEV)
    do = randn((Tq, H, d), seed + 3, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = forward_varlen(q, k, v, cuq, max(lens_q), causal=causal, scale=scale, cu_seqlens_k=cuk)
    dq, dk, dv = backward_varlen(q, k, v, o, lse, do, cuq, max(lens_q), causal=causal, scale=scale,
                                 deterministic=deterministic, cu_seqlens_k=cuk, max_seqlen_k=max(lens_k))
    torch.cuda.synchronize()
    check_device_status()
    if deterministic:
        again = backward_varlen(q, k, v, o, lse, do, cuq, max(lens_q), causal=causal, scale=scale,
                                deterministic=True, cu_seqlens_k=cuk, max_seqlen_k=max(lens_k))
        torch.cuda.synchronize()
        for a, b in zip((dq, dk, dv), again):
            assert torch.equal(a, b)
    g = H // Hkv
    ref = {"o": np.zeros((Tq, H, d)), "dq": np.zeros((Tq, H, d)), "dk": np.zeros((Tk, Hkv, d)),
           "dv": np.zeros((Tk, Hkv, d))}
    ref_lse = np.full((H, Tq), -np.inf)
    aq = ak = 0
    for nq, nk in zip(lens_q, lens_k):
        sq, sk = slice(aq, aq + nq), slice(ak, ak + nk)
        if nq > 0 and nk > 0:
            per = lambda t, sl, rep: np.repeat(to64(t[sl]).transpose(1, 0, 2)[None], rep, axis=1)
            ro, rl = oracle.fwd_rect(per(q, sq, 1), per(k, sk, g), per(v, sk, g), scale, causal=causal)
            r = oracle.bwd_rect(per(q, sq, 1), per(k, sk, g), per(v, sk, g), per(do, sq, 1), scale, causal=causal)
            ref["o"][sq] = ro[0].transpose(1, 0, 2)
            ref_lse[:, sq] = rl[0]
            ref["dq"][sq] = r["dq"][0].transpose(1, 0, 2)
            ref["dk"][sk] = r["dk"][0].reshape(Hkv, g, nk, d).sum(axis=1).transpose(1, 0, 2)
            ref["dv"][sk] = r["dv"][0].reshape(Hkv, g, nk, d).sum(axis=1).transpose(1, 0, 2)
        aq += nq
        ak += nk
    assert_o(to64(o), ref["o"])
    assert_lse(to64(lse), ref_lse)
    assert_grad(to64(dq), ref["dq"], "dQ")
    assert_grad(to64(dk), ref["dk"], "dK")
    assert_grad(to64(dv), ref["dv"], "dV")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_separate_key_ranges(d, causal):
    # more queries than keys, one query against many keys, an empty key range, an empty query range
    _case_kv([300, 1, 130, 0, 77], [200, 900, 0, 50, 301], 4, 2, d, causal, seed=131 + d)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_separate_key_ranges_deterministic(causal):
    _case_kv([500, 129, 64], [700, 129, 1000], 4, 1, 128, causal, seed=141, deterministic=True)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal,window", [(True, (100, 0)), (False, (64, 37)), (False, (-1, 20)), (True, (300, -1))])
def test_varlen_sliding_window_deterministic(d, causal, window):
    """The deterministic packed-window backward: d = 64 (128-query steps, so the
    first visitor of a query block is max(0, i * 128 - left) / 128) and d = 128
    (64-query steps), two-sided and one-sided windows."""
    _case([300, 1, 0, 129, 520, 64], 4, 2, d, causal, seed=171 + d + window[0], window=window, deterministic=True)


def test_varlen_separate_key_ranges_decode_mix():
    """A decode-like mix: 8 sequences with 1 .. 64 new queries against caches
    of up to 8192 keys (causal: the queries are each sequence's last
    positions), shared heads."""
    lens_q = [1, 64, 7, 33, 1, 16, 50, 2]
    lens_k = [8192, 4096, 1000, 3000, 129, 7777, 2048, 6000]
    _case_kv(lens_q, lens_k, 8, 2, 128, True, seed=181)
