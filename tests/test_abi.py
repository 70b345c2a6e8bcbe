"""CPU-side checks of the C ABI boundary: the library builds, loads without a
GPU, exports every function include/fa.h declares, and rejects bad arguments
on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

from exact_tiled_attention_10_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    path = fa_build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("fa_fwd", "fa_fwd_ex", "fa_bwd", "fa_bwd_ex", "fa_bwd_workspace_size",
                 "fa_quantize_fp8", "fa_fwd_fp8", "fa_check_device_status", "fa_last_error"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_signatures_cover_the_header():
    import exact_tiled_attention_10_gb300 as fa
    assert set(declared_functions()) == set(fa._SIGS)


def test_version_and_sizes(lib):
    lib.fa_version.restype = ctypes.c_int
    assert lib.fa_version() >= 1
    lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fa_bwd_workspace_size.argtypes = [ctypes.c_int] * 5
    # bf16: lse2 + D (B*H*Np floats each) + dQ accumulator (B*H*Np*d floats), Np = 384
    B, H, N, d = 2, 3, 300, 128
    Np = 384
    expect = 2 * (B * H * Np * 4) + B * H * Np * d * 4
    assert lib.fa_bwd_workspace_size(0, B, H, N, d) == expect
    assert lib.fa_bwd_workspace_size(0, B, H, N, 96) == 0
    lib.fa_fp8_num_blocks.restype = ctypes.c_int
    assert lib.fa_fp8_num_blocks(16384) == 256 and lib.fa_fp8_num_blocks(65) == 2


def _fwd(lib, q, k, v, o, lse, B, H, N, d, scale=0.125, causal=0):
    lib.fa_fwd.restype = ctypes.c_int
    lib.fa_fwd.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_int,
                                                                        ctypes.c_void_p, ctypes.c_void_p]
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, None, None)


def test_host_validation_without_gpu(lib):
    lib.fa_last_error.restype = ctypes.c_char_p
    A = 4096  # a 16-byte aligned fake address: validation rejects before any use
    # null pointer
    assert _fwd(lib, None, A, A, A, A, 1, 1, 128, 64) == 1
    assert b"q must not be NULL" in lib.fa_last_error()
    # misaligned pointer
    assert _fwd(lib, A + 2, A, A, A, A, 1, 1, 128, 64) == 1
    assert b"aligned" in lib.fa_last_error()
    # bad sizes
    assert _fwd(lib, A, A, A, A, A, 0, 1, 128, 64) == 1
    assert _fwd(lib, A, A, A, A, A, 1, 1, -5, 64) == 1
    # unsupported head dim
    assert _fwd(lib, A, A, A, A, A, 1, 1, 128, 96) == 2
    # non-finite scale
    assert _fwd(lib, A, A, A, A, A, 1, 1, 128, 64, scale=float("nan")) == 1


def test_binding_refuses_cpu_tensors():
    import torch
    import exact_tiled_attention_10_gb300 as fa
    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.forward(x, x, x)
