"""Unwritten-output checks: every tensor the Python binding allocates (outputs,
LSE, workspaces) is filled with NaN (bytes with 0xFF) before the kernels run,
and every entry point must then produce no NaN and the same results as a run
on fresh memory.  A row the kernels forget to write, or scratch they read
before initialising, shows up as NaN or as a difference; zero-filled memory
would hide it, since fully masked rows are zero by definition (the attention
wiki's fully-masked-row convention: O = 0, LSE = -inf, zero gradients).
Cases include fully masked rows (kv_len 0), empty sequences and block
lists, query rows that see no key, ragged lengths and split keys."""
import math

import pytest
import torch

import exact_tiled_attention_10_gb300 as fa
from exact_tiled_attention_10_gb300.inputs import randn

pytestmark = pytest.mark.gpu
DEV = "cuda"


class _PoisonTorch:
    """torch, except that empty / empty_like return NaN-filled (0xFF-filled)
    tensors."""

    def __getattr__(self, name):
        return getattr(torch, name)

    @staticmethod
    def _fill(t):
        if t.is_floating_point():
            t.fill_(float("nan"))
        elif t.dtype == torch.uint8:
            t.fill_(0xFF)
        else:
            t.fill_(-1)
        return t

    def empty(self, *a, **k):
        return self._fill(torch.empty(*a, **k))

    def empty_like(self, *a, **k):
        return self._fill(torch.empty_like(*a, **k))


def _no_nan(*ts):
    for t in ts:
        assert not torch.isnan(t.float()).any(), "NaN left in an output of shape %s" % (tuple(t.shape),)


def _same(a, b, exact=True):
    for x, y in zip(a, b):
        if exact:
            assert torch.equal(x, y)
        else:
            tol = 1e-2 * max(y.float().abs().max().item(), 1e-6)
            assert (x.float() - y.float()).abs().max().item() <= tol


def _run_both(monkeypatch, fn, exact=True):
    ref = fn()
    torch.cuda.synchronize()
    with monkeypatch.context() as m:
        m.setattr(fa, "torch", _PoisonTorch())
        got = fn()
        torch.cuda.synchronize()
    fa.check_device_status()
    _no_nan(*got)
    _same(got, ref, exact)
    return got


def _qkv(B, H, Hkv, N, d, seed, Nk=None):
    Nk = N if Nk is None else Nk
    return (randn((B, H, N, d), seed, device=DEV), randn((B, Hkv, Nk, d), seed + 1, device=DEV),
            randn((B, Hkv, Nk, d), seed + 2, device=DEV), randn((B, H, N, d), seed + 3, device=DEV))


@pytest.mark.parametrize("d", [64, 128])
def test_plain_forward_backward_with_empty_rows(monkeypatch, d):
    q, k, v, do = _qkv(2, 4, 4, 200, d, 11)
    kv = torch.tensor([0, 77], dtype=torch.int32, device=DEV)
    o, lse = _run_both(monkeypatch, lambda: fa.forward(q, k, v, causal=True, kv_lens=kv))
    assert (lse[0] == -math.inf).all() and (o[0] == 0).all()
    _run_both(monkeypatch, lambda: fa.backward(q, k, v, o, lse, do, causal=True, kv_lens=kv)[1:])
    _run_both(monkeypatch, lambda: fa.backward(q, k, v, o, lse, do, causal=True, kv_lens=kv)[:1], exact=False)


def test_split_forward(monkeypatch):
    q, k, v, _ = _qkv(1, 2, 2, 700, 128, 13)
    _run_both(monkeypatch, lambda: fa.forward_split(q, k, v, num_splits=3))


def test_grouped_backward_with_split_units(monkeypatch):
    q, k, v, do = _qkv(1, 8, 2, 300, 128, 15)
    o, lse = fa.forward(q, k, v, causal=True)
    _run_both(monkeypatch, lambda: fa.backward(q, k, v, o, lse, do, causal=True)[1:])


def test_window(monkeypatch):
    q, k, v, do = _qkv(1, 4, 2, 600, 128, 17)
    o, lse = _run_both(monkeypatch, lambda: fa.forward(q, k, v, window=(64, 0)))
    _run_both(monkeypatch, lambda: fa.backward(q, k, v, o, lse, do, window=(64, 0))[1:])


def test_block_sparse_with_an_empty_list(monkeypatch):
    q, k, v, do = _qkv(1, 2, 2, 384, 128, 19)
    mask = torch.tensor([[1, 0, 0], [0, 0, 0], [1, 1, 1]], dtype=torch.bool)
    rp, ci = fa.block_lists(mask, DEV)
    o, lse = _run_both(monkeypatch, lambda: fa.forward_block_sparse(q, k, v, rp, ci))
    assert (lse[:, :, 128:256] == -math.inf).all()
    _run_both(monkeypatch, lambda: fa.backward_block_sparse(q, k, v, o, lse, do, rp, ci)[1:])


def test_rect_decode_and_more_queries_than_keys(monkeypatch):
    q, k, v, _ = _qkv(2, 8, 2, 1, 128, 21, Nk=5000)
    _run_both(monkeypatch, lambda: fa.forward_rect(q, k, v, causal=True))
    q, k, v, do = _qkv(1, 2, 2, 300, 128, 23, Nk=100)
    o, lse = _run_both(monkeypatch, lambda: fa.forward_rect(q, k, v, causal=True))
    _run_both(monkeypatch, lambda: fa.backward_rect(q, k, v, o, lse, do, causal=True)[1:])


def test_varlen_with_an_empty_sequence(monkeypatch):
    lens = [130, 0, 77]
    T = sum(lens)
    cu = torch.tensor([0, 130, 130, 207], dtype=torch.int32, device=DEV)
    q, k, v, do = (randn((T, 4, 128), 25 + i, device=DEV) for i in range(4))
    o, lse = _run_both(monkeypatch, lambda: fa.forward_varlen(q, k, v, cu, max(lens), causal=True))
    _run_both(monkeypatch, lambda: fa.backward_varlen(q, k, v, o, lse, do, cu, max(lens), causal=True)[1:])
    _run_both(monkeypatch,
              lambda: fa.backward_varlen(q, k, v, o, lse, do, cu, max(lens), causal=True, deterministic=True))


def test_bnhd(monkeypatch):
    q, k, v, do = (randn((2, 130, 4, 64), 27 + i, device=DEV) for i in range(4))
    o, lse = _run_both(monkeypatch, lambda: fa.forward_bnhd(q, k, v, causal=True))
    _run_both(monkeypatch, lambda: fa.backward_bnhd(q, k, v, o, lse, do, causal=True)[1:])


def test_deterministic_backward(monkeypatch):
    q, k, v, do = _qkv(2, 4, 2, 300, 128, 29)
    kv = torch.tensor([0, 300], dtype=torch.int32, device=DEV)
    o, lse = fa.forward(q, k, v, causal=True, kv_lens=kv)
    _run_both(monkeypatch, lambda: fa.backward(q, k, v, o, lse, do, causal=True, kv_lens=kv, deterministic=True))


def test_fp8_quantiser_and_forward(monkeypatch):
    q, k, v, _ = _qkv(1, 2, 2, 200, 128, 31)
    q8, sq, k8, sk, v8, sv = _run_both(monkeypatch,
                                       lambda: tuple(t for pair in fa.quantize_fp8_qkv(q, k, v) for t in pair))
    _run_both(monkeypatch, lambda: fa.forward_fp8(q8, k8, v8, sq, sk, sv))


def test_varlen_separate_key_ranges(monkeypatch):
    """Separate query / key ranges, one sequence with keys but no queries:
    its dK, dV rows must be written (zero)."""
    lens_q, lens_k = [130, 0, 77], [60, 50, 200]
    cuq = torch.tensor([0, 130, 130, 207], dtype=torch.int32, device=DEV)
    cuk = torch.tensor([0, 60, 110, 310], dtype=torch.int32, device=DEV)
    q, do = (randn((207, 4, 128), 41 + i, device=DEV) for i in range(2))
    k, v = (randn((310, 2, 128), 43 + i, device=DEV) for i in range(2))
    o, lse = _run_both(monkeypatch, lambda: fa.forward_varlen(q, k, v, cuq, 130, causal=True, cu_seqlens_k=cuk))
    dq, dk, dv = _run_both(monkeypatch, lambda: fa.backward_varlen(q, k, v, o, lse, do, cuq, 130, causal=True,
                                                                   cu_seqlens_k=cuk, max_seqlen_k=200,
                                                                   deterministic=True))
    assert (dk[60:110] == 0).all() and (dv[60:110] == 0).all()


def test_fp8_backward(monkeypatch):
    """The FP8 backward's dQ, dK, dV (float32), its workspace (dO codes and
    scales, transposed K codes, statistics, dQ accumulator) all poisoned."""
    q, k, v, do = _qkv(2, 2, 2, 300, 128, 33)
    (q8, sq), (k8, sk), (v8, sv) = fa.quantize_fp8_qkv(q, k, v)
    kv = torch.tensor([0, 250], dtype=torch.int32, device=DEV)
    o, lse = fa.forward_fp8(q8, k8, v8, sq, sk, sv, causal=True, kv_lens=kv)
    _run_both(monkeypatch, lambda: fa.backward_fp8(q8, k8, v8, sq, sk, sv, o, lse, do, causal=True, kv_lens=kv)[1:])
    _run_both(monkeypatch, lambda: fa.backward_fp8(q8, k8, v8, sq, sk, sv, o, lse, do, causal=True,
                                                   kv_lens=kv)[:1], exact=False)
