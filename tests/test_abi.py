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


def test_split_plan_without_gpu(lib):
    """Split-key plan (fa_fwd_split_count / _workspace_size) for a 152-SM
    device (the default when no GPU is visible).  Long_head (B=2 H=16 N=4096)
    and long_seq (B=1 H=8 N=16384) both have 512 items of 256 query rows: 3
    full rounds of 152 plus 56; splitting those 56 into 2 key ranges makes the
    last round half as long (estimated 120 vs 136 key blocks, resp. 456 vs 520),
    so 56 * 2 = 112 partials of 256 rows x (128 + 1) float32 values."""
    cnt, wsz = lib.fa_fwd_split_count, lib.fa_fwd_split_workspace_size
    cnt.restype, cnt.argtypes = ctypes.c_int, [ctypes.c_int] * 7
    wsz.restype, wsz.argtypes = ctypes.c_size_t, [ctypes.c_int] * 7
    expect = 112 * 256 * 128 * 4 + 112 * 256 * 4
    for (B, H, N) in ((2, 16, 4096), (1, 8, 16384)):
        assert cnt(B, H, N, 128, 0, 0, 0) == 2
        assert wsz(B, H, N, 128, 0, 0, 0) == expect
        assert cnt(B, H, N, 128, 1, 0, 0) == 1      # causal: not split automatically
        assert cnt(B, H, N, 128, 0, 1, 0) == 1      # key-padded: not split automatically
        assert wsz(B, H, N, 128, 1, 0, 0) == 0
    assert cnt(1, 1, 128, 64, 0, 0, 0) == 1         # one key block
    assert cnt(2, 2, 300, 64, 0, 0, 1) == 1         # explicit: no split
    assert cnt(2, 2, 300, 64, 1, 0, 3) == 3         # explicit: every item in 3 ranges
    assert wsz(2, 2, 300, 64, 1, 0, 3) == (2 * 2 * 2) * 3 * 256 * (64 + 1) * 4
    assert cnt(2, 2, 300, 64, 0, 0, 1000) == 64     # capped
    assert wsz(2, 2, 300, 64, 0, 0, -1) == 0


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


def _prototype_arity():
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"\b(fa_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", src):
        args = m.group(2).strip()
        out[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    return out


def test_binding_argument_counts_match_the_prototypes():
    import exact_tiled_attention_10_gb300 as fa
    arity = _prototype_arity()
    for name, (argtypes, _) in fa._SIGS.items():
        assert name in arity, name
        assert len(argtypes) == arity[name], (name, len(argtypes), arity[name])


def test_host_validation_of_the_variant_entry_points():
    """Bad arguments of the window, block-sparse, rectangular, grouped and
    fused-quantiser entry points are refused on the host, before any CUDA
    call (so this runs without a GPU)."""
    import exact_tiled_attention_10_gb300 as fa
    lib = fa.load_library()
    A = 4096
    # window: an edge below -1, heads not a multiple of the key/value heads
    assert lib.fa_fwd_window(A, A, A, A, A, 1, 4, 4, 256, 128, 0.1, 0, -2, 5, None, None) == 1
    assert lib.fa_fwd_window(A, A, A, A, A, 1, 4, 3, 256, 128, 0.1, 0, 5, 5, None, None) == 1
    # [B, N, H, d] layout: bad group, unsupported head dim, B * N beyond 32 bits, workspace too small
    assert lib.fa_fwd_bnhd(A, A, A, A, A, 2, 256, 4, 3, 128, 0.1, 0, None) == 1
    assert lib.fa_fwd_bnhd(A, A, A, A, A, 2, 256, 4, 4, 96, 0.1, 0, None) == 2
    assert lib.fa_fwd_bnhd(A, A, A, A, A, 1 << 16, 1 << 16, 4, 4, 128, 0.1, 0, None) == 1
    assert lib.fa_bwd_bnhd_workspace_size(2, 256, 4, 128) == lib.fa_bwd_varlen_workspace_size(2, 256, 4, 128) > 0
    assert lib.fa_bwd_bnhd(A, A, A, A, A, A, A, A, A, 2, 256, 4, 4, 128, 0.1, 0, A, 1024, None) == 1
    # packed sliding window: bad edge; separate key ranges: missing offsets, a window with them
    assert lib.fa_fwd_varlen_window(A, A, A, A, A, A, 2, 512, 256, 4, 4, 128, 0.1, 0, -2, 0, None) == 1
    assert lib.fa_fwd_varlen_kv(A, A, A, A, A, A, None, 2, 512, 512, 256, 4, 4, 128, 0.1, 0, None) == 1
    assert lib.fa_bwd_varlen_kv_workspace_size(2, 256, 300, 4, 3, 128, 0) == 0
    assert (lib.fa_bwd_varlen_kv_workspace_size(2, 256, 300, 4, 2, 128, 1) >
            lib.fa_bwd_varlen_kv_workspace_size(2, 256, 300, 4, 2, 128, 0) > 0)
    # FP8 with shared heads: bad group
    assert lib.fa_fwd_fp8_gqa(A, A, A, A, A, A, A, A, 1, 4, 3, 256, 128, 0.1, 0, None, None) == 1
    # deterministic packed / [B, N, H, d]: more workspace than the default; bad group
    assert lib.fa_bwd_varlen_deterministic_workspace_size(3, 300, 8, 2, 128) > lib.fa_bwd_varlen_workspace_size(3, 300, 8, 128)
    assert lib.fa_bwd_bnhd_deterministic_workspace_size(2, 256, 4, 3, 128) == 0
    assert lib.fa_bwd_varlen_deterministic(A, A, A, A, A, A, A, A, A, None, 2, 512, 256, 4, 4, 128, 0.1, 0, A, 1 << 30,
                                           None) == 1
    # block-sparse: missing lists, workspace too small
    assert lib.fa_fwd_block_sparse(A, A, A, A, A, 1, 4, 4, 256, 128, 0.1, 0, None, A, None, None) == 1
    need = lib.fa_bwd_block_sparse_workspace_size(1, 4, 256, 128)
    assert need > lib.fa_bwd_workspace_size(0, 1, 4, 256, 128)
    assert lib.fa_bwd_block_sparse(A, A, A, A, A, A, A, A, A, 1, 4, 4, 256, 128, 0.1, 0, A, A, None, A, need - 1,
                                   None) == 1
    # rectangular: no keys, bad group, negative split count
    assert lib.fa_fwd_rect(A, A, A, A, A, 1, 4, 4, 1, 0, 128, 0.1, 1, None, 0, None, 0, None) == 1
    assert lib.fa_fwd_rect(A, A, A, A, A, 1, 4, 3, 1, 100, 128, 0.1, 1, None, 0, None, 0, None) == 1
    assert lib.fa_fwd_rect(A, A, A, A, A, 1, 4, 4, 1, 100, 128, 0.1, 1, None, -1, None, 0, None) == 1
    assert lib.fa_fwd_rect_workspace_size(1, 4, 3, 1, 100, 128, 0) == 0
    # a decode step (one query per head, long cache) is split; a long prefill is not
    assert lib.fa_fwd_rect_split_count(1, 32, 8, 1, 131072, 128, 0) > 1
    assert lib.fa_fwd_rect_split_count(8, 32, 8, 4096, 4096, 128, 0) == 1
    # fused quantiser: bad group
    assert lib.fa_quantize_fp8_qkv(A, A, A, A, A, A, A, A, A, 1, 4, 3, 256, 128, None) == 1
    # grouped backward: the split workspace is larger only when key blocks are few
    assert lib.fa_bwd_gqa_workspace_size(2, 16, 2, 4096, 128) > lib.fa_bwd_workspace_size(0, 2, 16, 4096, 128)
    assert lib.fa_bwd_gqa_workspace_size(64, 16, 16, 4096, 128) <= lib.fa_bwd_workspace_size(0, 64, 16, 4096, 128) + 256


def test_deterministic_backward_workspace_without_gpu():
    """fa_bwd_deterministic_workspace_size: fa_bwd's layout, then A - 1 more
    float32 dQ accumulators and A x 4 turn counters per dQ tile, where
    A = min(8, key blocks, ceil(152 / (B * Hkv)) + 1) depends on the shape
    only; argument errors are caught on the host."""
    import exact_tiled_attention_10_gb300 as fa
    lib = fa.load_library()
    size = lib.fa_bwd_deterministic_workspace_size
    for (B, H, Hkv, N, d) in [(2, 16, 16, 4096, 128), (1, 8, 1, 300, 64), (64, 16, 16, 1024, 128)]:
        Np = -(-N // 128) * 128
        kt = -(-N // 128)
        A = min(8, kt, -(-152 // (B * Hkv)) + 1)
        acc = B * H * Np * d * 4
        turns = A * B * H * (Np // (64 if d == 128 else 128)) * 4 * 4
        assert size(B, H, Hkv, N, d) == lib.fa_bwd_workspace_size(0, B, H, N, d) + (A - 1) * acc + turns
    assert size(1, 8, 3, 256, 128) == 0 and size(1, 8, 8, 256, 96) == 0
    A_ = 4096
    need = size(1, 4, 4, 256, 128)
    # bad group; workspace below fa_bwd's own layout
    assert lib.fa_bwd_deterministic(A_, A_, A_, A_, A_, A_, A_, A_, A_, 1, 4, 3, 256, 128, 0.1, 0, None, A_, need,
                                    None) == 1
    assert lib.fa_bwd_deterministic(A_, A_, A_, A_, A_, A_, A_, A_, A_, 1, 4, 4, 256, 128, 0.1, 0, None, A_, 1024,
                                    None) == 1
