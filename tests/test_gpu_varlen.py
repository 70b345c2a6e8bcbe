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
from parity_util import O_TOL, assert_close_abs, assert_grad, assert_lse, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(lens, H, Hkv, d, causal, seed, deterministic=False):
    T = int(sum(lens))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=DEV)
    q = randn((T, H, d), seed, device=DEV)
    k = randn((T, Hkv, d), seed + 1, device=DEV)
    v = randn((T, Hkv, d), seed + 2, device=DEV)
    do = randn((T, H, d), seed + 3, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = forward_varlen(q, k, v, cu, max(lens), causal=causal, scale=scale)
    dq, dk, dv = backward_varlen(q, k, v, o, lse, do, cu, max(lens), causal=causal, scale=scale,
                                 deterministic=deterministic)
    torch.cuda.synchronize()
    check_device_status()
    g = H // Hkv
    # reference, one sequence at a time
    ref = {n: np.zeros(t.shape) for n, t in (("o", q), ("dq", q), ("dk", k), ("dv", v))}
    ref_lse = np.zeros((H, T))
    a = 0
    for n in lens:
        if n > 0:
            sl = slice(a, a + n)
            per = lambda t, rep: np.repeat(to64(t[sl]).transpose(1, 0, 2)[None], rep, axis=1)
            r = oracle.bwd(per(q, 1), per(k, g), per(v, g), per(do, 1), scale, causal=causal)
            ref["o"][sl] = r["o"][0].transpose(1, 0, 2)
            ref["dq"][sl] = r["dq"][0].transpose(1, 0, 2)
            ref["dk"][sl] = r["dk"][0].reshape(Hkv, g, n, d).sum(axis=1).transpose(1, 0, 2)
            ref["dv"][sl] = r["dv"][0].reshape(Hkv, g, n, d).sum(axis=1).transpose(1, 0, 2)
            ref_lse[:, sl] = r["lse"][0]
        a += n
    assert_close_abs(to64(o), ref["o"], O_TOL, "O")
    assert_lse(to64(lse), ref_lse)
    assert_grad(to64(dq), ref["dq"], "dQ")
    assert_grad(to64(dk), ref["dk"], "dK")
    assert_grad(to64(dv), ref["dv"], "dV")


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
