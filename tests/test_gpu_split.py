"""GPU parity of the split-key forward (chapter 18 §18.8.2, FlashDecoding):
each (head, 256-row) item's key sequence is cut into contiguous ranges that
separate work units compute, and a second kernel merges the ranges' outputs
with their log-sum-exp weights.  The result must match the oracle like the
unsplit forward, for explicit range counts (including more ranges than key
blocks, i.e. empty ranges, and key padding that empties whole ranges), for
the automatic plan, and for the FP8 forward."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_10_gb300 import (check_device_status, forward, forward_fp8, forward_fp8_split,
                                            forward_split, quantize_fp8, split_count)
from exact_tiled_attention_10_gb300.inputs import WORKLOADS, qkv
from parity_util import FP8_O_TOL, O_TOL, assert_close_abs, assert_lse, sample_rows, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check_split(B, H, N, d, causal, splits, kv=None, seed=11):
    q, k, v = qkv(B, H, N, d, seed, device=DEV, with_dout=False)
    kvd = None if kv is None else torch.tensor(kv, dtype=torch.int32, device=DEV)
    o, lse = forward_split(q, k, v, causal=causal, kv_lens=kvd, num_splits=splits)
    torch.cuda.synchronize()
    check_device_status()
    kvn = None if kv is None else np.asarray(kv, dtype=np.int32)
    ref_o, ref_l = oracle.fwd(to64(q), to64(k), to64(v), 1 / math.sqrt(d), causal=causal, kv_lens=kvn)
    assert_close_abs(to64(o), ref_o, O_TOL, "O (%d ranges)" % splits)
    assert_lse(to64(lse), ref_l, what="LSE (%d ranges)" % splits)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,splits", [(200, 2), (383, 3), (520, 5), (1000, 4)])
def test_split_ranges_match_oracle(d, causal, N, splits):
    _check_split(2, 2, N, d, causal, splits, seed=N + d)


@pytest.mark.parametrize("causal", [False, True])
def test_split_with_key_padding_and_empty_ranges(causal):
    # kv_len 0: every range empty; kv_len 1 and 65: one key block, so the
    # later ranges of those items hold no key
    _check_split(6, 2, 300, 128, causal, 3, kv=[0, 1, 65, 129, 300, 300], seed=5)


def test_more_ranges_than_key_blocks():
    _check_split(1, 3, 150, 64, False, 5, seed=6)


def test_one_range_is_the_unsplit_forward():
    q, k, v = qkv(2, 4, 1000, 128, 12, device=DEV, with_dout=False)
    o1, l1 = forward(q, k, v, causal=True)
    o2, l2 = forward_split(q, k, v, causal=True, num_splits=1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_automatic_plan_long_head_noncausal():
    """long_head non-causal: 512 items; on a 152-SM GB300 the plan keeps 456
    whole and splits the last 56 in two (items 456..511: query pairs 8..15 of
    head 28 and all of heads 29..31).  Rows of heads 28 and 31 are compared
    with the oracle, everything with the unsplit forward."""
    w = WORKLOADS["long_head"]
    q, k, v = qkv(w.B, w.H, w.N, w.d, w.seed, device=DEV, with_dout=False)
    S = split_count(w.B, w.H, w.N, w.d, causal=False)
    o, lse = forward_split(q, k, v, causal=False)
    o1, l1 = forward(q, k, v, causal=False)
    torch.cuda.synchronize()
    check_device_status()
    assert S >= 1
    assert (o.float() - o1.float()).abs().max().item() <= O_TOL
    assert (lse - l1).abs().max().item() <= 1e-3
    for bh in (28, 31):
        b, h = divmod(bh, w.H)
        rows = np.concatenate([sample_rows(w.N, 24, seed=bh)[:12], np.arange(2048, 4096, 171)])
        ref_o, ref_l = oracle.fwd_rows(to64(q[b, h]), to64(k[b, h]), to64(v[b, h]), w.scale, False, w.N, rows)
        assert_close_abs(to64(o[b, h, rows]), ref_o, O_TOL, "O[%d,%d]" % (b, h))
        assert_lse(to64(lse[b, h, rows]), ref_l, what="LSE[%d,%d]" % (b, h))


@pytest.mark.parametrize("splits", [0, 3])
def test_fp8_split_matches_unsplit_fp8(splits):
    """The FP8 forward split into key ranges: O and LSE agree with the unsplit
    FP8 forward (same quantised operands) within the FP8 tolerance, and O
    with the oracle on the original inputs."""
    B, H, N = 2, 2, 2048
    q, k, v = qkv(B, H, N, 128, 33, device=DEV, with_dout=False)
    (q8, sq), (k8, sk), (v8, sv) = (quantize_fp8(t) for t in (q, k, v))
    o, lse = forward_fp8_split(q8, k8, v8, sq, sk, sv, causal=False, num_splits=splits)
    o1, l1 = forward_fp8(q8, k8, v8, sq, sk, sv, causal=False)
    torch.cuda.synchronize()
    check_device_status()
    assert (o.float() - o1.float()).abs().max().item() <= FP8_O_TOL
    assert (lse - l1).abs().max().item() <= 1e-3
    ref_o, _ = oracle.fwd(to64(q), to64(k), to64(v), 1 / math.sqrt(128))
    assert_close_abs(to64(o), ref_o, FP8_O_TOL, "FP8 O (%d ranges)" % splits)
