"""GPU parity of block-sparse attention (chapter 18 §18.8.1: for each query
block the list of key blocks to compute; every other block is skipped).

Blocks are 128 x 128.  The oracle applies the same block mask element by
element on the materialised S.  Cases: random masks of several densities,
lists whose two 128-row tiles of one work item use disjoint and interleaved
blocks (the merged K/V stream then has blocks only one tile uses), empty
lists (fully masked rows), the all-ones and diagonal masks, the causal and
key-padding masks, shared key/value heads, ragged N, and a long sequence on
sampled rows and keys.  O is held to the flat 1e-2 except on rows that see
fewer than 16 keys (the first rows of a causal diagonal block when it is the
row's only block), which are held to the worst case of the kernel's two
bf16 roundings (parity_util.assert_o)."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_10_gb300 import (backward_block_sparse, block_lists, check_device_status, forward,
                                            forward_block_sparse)
from exact_tiled_attention_10_gb300.inputs import qkv
from parity_util import assert_close_abs, assert_grad, assert_lse, assert_o, rounding_context, sample_rows, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(B, H, Hkv, N, d, causal, bm, kv=None, seed=5, deterministic=False):
    q, _, _, do = qkv(B, H, N, d, seed, device=DEV)
    _, k, v = qkv(B, Hkv, N, d, seed + 50, device=DEV, with_dout=False)
    kvd = None if kv is None else torch.tensor(kv, dtype=torch.int32, device=DEV)
    rp, ci = block_lists(bm, DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = forward_block_sparse(q, k, v, rp, ci, causal=causal, scale=scale, kv_lens=kvd)
    dq, dk, dv = backward_block_sparse(q, k, v, o, lse, do, rp, ci, causal=causal, scale=scale, kv_lens=kvd,
                                       deterministic=deterministic)
    torch.cuda.synchronize()
    check_device_status()
    if deterministic:  # a second run agrees bit for bit
        again = backward_block_sparse(q, k, v, o, lse, do, rp, ci, causal=causal, scale=scale, kv_lens=kvd,
                                      deterministic=True)
        torch.cuda.synchronize()
        for a, b in zip((dq, dk, dv), again):
            assert torch.equal(a, b)
    g = H // Hkv
    kvn = None if kv is None else np.asarray(kv, dtype=np.int32)
    kr, vr = np.repeat(to64(k), g, axis=1), np.repeat(to64(v), g, axis=1)
    bma = np.asarray(bm)
    ref = oracle.bwd(to64(q), kr, vr, to64(do), scale, causal=causal, kv_lens=kvn, block_mask=bma, block_size=128)
    nvis, absref = rounding_context(
        lambda qq, vv: oracle.fwd(qq, kr, vv, scale, causal=causal, kv_lens=kvn, block_mask=bma, block_size=128),
        to64(q), vr)
    assert_o(to64(o), ref["o"], nvis=nvis, absref=absref)
    assert_lse(to64(lse), ref["lse"])
    assert_grad(to64(dq), ref["dq"], "dQ")
    assert_grad(to64(dk), ref["dk"].reshape(B, Hkv, g, N, d).sum(axis=2), "dK")
    assert_grad(to64(dv), ref["dv"].reshape(B, Hkv, g, N, d).sum(axis=2), "dV")


def _random_mask(nb, density, seed):
    rng = np.random.default_rng(seed)
    return (rng.random((nb, nb)) < density).astype(np.uint8)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("density", [0.3, 0.7])
def test_random_block_masks(d, causal, density):
    N = 600  # 5 blocks, the last ragged
    bm = _random_mask(5, density, seed=int(density * 10) + d + causal)
    _case(2, 2, 2, N, d, causal, bm, seed=11 + d)


def test_interleaved_and_disjoint_tile_lists():
    """Query blocks 0/1 (one work item) use blocks {0, 2, 4} / {1, 3}; blocks
    2/3 use {3} / {0, 4}; block 4 has no list (rows fully masked)."""
    bm = np.zeros((5, 5), dtype=np.uint8)
    for i, cols in enumerate([[0, 2, 4], [1, 3], [3], [0, 4], []]):
        bm[i, cols] = 1
    for d in (64, 128):
        _case(1, 2, 2, 640, d, False, bm, seed=17 + d)


def test_block_sparse_with_padding_and_shared_heads():
    bm = _random_mask(4, 0.5, seed=3)
    bm[:, 0] = 1
    _case(3, 4, 2, 500, 128, True, bm, kv=[0, 200, 500], seed=23)
    _case(2, 4, 1, 389, 64, False, bm, kv=[77, 389], seed=29)


def test_all_ones_mask_equals_dense_forward():
    q, k, v = qkv(2, 2, 700, 128, 31, device=DEV, with_dout=False)
    rp, ci = block_lists(np.ones((6, 6)), DEV)
    for causal in (False, True):
        o1, l1 = forward(q, k, v, causal=causal)
        o2, l2 = forward_block_sparse(q, k, v, rp, ci, causal=causal)
        torch.cuda.synchronize()
        assert_close_abs(to64(o2), to64(o1), 2e-3, "O (all blocks vs dense)")
        assert_lse(to64(l2), to64(l1), 1e-4)


def test_block_sparse_long_sequence_sampled():
    """N = 8192, d = 128, causal, a random mask of density 0.25 plus the
    diagonal: sampled rows and keys of two heads against the row-sampled
    oracle."""
    B, H, N, d = 1, 4, 8192, 128
    nb = N // 128
    bm = _random_mask(nb, 0.25, seed=41)
    np.fill_diagonal(bm, 1)
    q, k, v, do = qkv(B, H, N, d, 47, device=DEV)
    rp, ci = block_lists(bm, DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = forward_block_sparse(q, k, v, rp, ci, causal=True, scale=scale)
    dq, dk, dv = backward_block_sparse(q, k, v, o, lse, do, rp, ci, causal=True, scale=scale)
    torch.cuda.synchronize()
    check_device_status()
    rows = sorted(set(sample_rows(N, 24, seed=5)))
    keys = sorted(set(sample_rows(N, 12, seed=6)))
    for h in (0, 3):
        qh, kh, vh, gh = (to64(t[0, h]) for t in (q, k, v, do))
        run = lambda qq, vv: oracle.fwd_rows(qq, kh, vv, scale, True, N, rows, block_mask=bm, block_size=128)
        o_ref, lse_ref = run(qh, vh)
        nvis, absref = rounding_context(run, qh, vh)
        assert_o(to64(o[0, h])[rows], o_ref, "O rows", nvis=nvis, absref=absref)
        assert_lse(to64(lse[0, h])[rows], lse_ref)
        # gradient scale: the oracle's max-abs over the sampled rows / keys
        g = oracle.bwd_rows(qh, kh, vh, gh, scale, True, N, rows, keys, block_mask=bm, block_size=128)
        assert_grad(to64(dq[0, h])[rows], g["dq"], "dQ rows")
        assert_grad(to64(dk[0, h])[keys], g["dk"], "dK keys")
        assert_grad(to64(dv[0, h])[keys], g["dv"], "dV keys")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_block_sparse_deterministic(d, causal):
    """The deterministic backward with block lists: a key block's turn is its
    place in the query block's list (binary search); parity with the oracle,
    shared heads, key lengths, and a bitwise repeat."""
    N = 1300
    nb = (N + 127) // 128
    rng = np.random.default_rng(97 + d + causal)
    bm = (rng.random((nb, nb)) < 0.45).astype(np.uint8)
    bm[:, 0] = 1
    bm[3] = 0  # an empty list
    _case(2, 4, 2, N, d, causal, bm, kv=[N, 900], seed=101 + d, deterministic=True)
