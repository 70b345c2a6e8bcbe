"""The allocation-free backward (fa_bwd_noalloc) against the regular one.

fa_bwd_noalloc serves callers that cannot allocate device memory (a plugin
inside a framework that owns the whole device-memory pool, a runtime that
forbids allocation after start-up): its scratch is a fixed array of device
memory inside the library instead of a caller workspace.  This test calls both
entry points through the C ABI on the same inputs and requires the same
gradients within the tolerance of the parity tests, on two calls in a row (the
second call finds the first call's leftovers in the shared array).  It is
named to be collected last and runs the same alone or after the other tests.
"""
import ctypes
import math

import pytest
import torch

import exact_tiled_attention_10_gb300 as fa
from exact_tiled_attention_10_gb300.inputs import qkv

pytestmark = pytest.mark.gpu
GRAD_REL_TOL = 2e-2


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
def test_noalloc_backward_matches_workspace_backward_twice(d, causal):
    lib = fa.load_library()
    B, H, N = 2, 4, 1000
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = qkv(B, H, N, d, 77 + d, device="cuda")
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    # reference: the existing entry point with a caller workspace
    wsz = lib.fa_bwd_workspace_size(B, H, N, d)
    assert 0 < wsz <= lib.fa_bwd_noalloc_max_scratch()
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    ref = [torch.empty_like(q) for _ in range(3)]
    st = lib.fa_bwd(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(do), _p(ref[0]), _p(ref[1]), _p(ref[2]),
                    B, H, N, d, ctypes.c_float(scale), int(causal), None, _p(ws), ctypes.c_size_t(wsz), stream)
    assert st == 0, lib.fa_last_error()

    for call in range(2):
        out = [torch.full_like(q, float("nan")) for _ in range(3)]
        st = lib.fa_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(do), _p(out[0]), _p(out[1]),
                                _p(out[2]), B, H, N, d, ctypes.c_float(scale), int(causal), None, stream)
        assert st == 0, lib.fa_last_error()
        torch.cuda.synchronize()
        fa.check_device_status()
        for name, a, r in zip(("dQ", "dK", "dV"), out, ref):
            assert torch.isfinite(a.float()).all(), (call, name)
            err = (a.float() - r.float()).abs().max().item()
            tol = GRAD_REL_TOL * r.float().abs().max().item()
            assert err <= tol, "call %d %s: %.3e > %.3e" % (call, name, err, tol)


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = fa.load_library()
    cap = lib.fa_bwd_noalloc_max_scratch()
    B, H, N, d = 64, 64, 4096, 128
    assert lib.fa_bwd_workspace_size(B, H, N, d) > cap
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")  # never touched: rejected before launch
    lse = torch.empty(16, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.fa_bwd_noalloc(_p(x), _p(x), _p(x), _p(x), _p(lse), _p(x), _p(x), _p(x), _p(x), B, H, N, d,
                            ctypes.c_float(0.1), 0, None, stream)
    assert st == fa.FA_ERR_INVALID_ARG
    assert b"static" in lib.fa_last_error()
