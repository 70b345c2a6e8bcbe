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
    for must in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_quantize_fp8", "fa_fwd_fp8",
                 "fa_check_device_status", "fa_last_error", "fa_attn_params_init", "fa_attn_fwd",
                 "fa_attn_bwd", "fa_attn_fwd_workspace_size", "fa_attn_bwd_workspace_size"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_exports_nothing_else():
    """The shared library's exported functions are exactly the header's (the
    variant implementations behind fa_attn_fwd / fa_attn_bwd are hidden)."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    path = fa_build.build()
    out = subprocess.run([nm, "-D", "--defined-only", path], check=True, capture_output=True, text=True).stdout
    exported = sorted(set(l.split()[-1] for l in out.splitlines() if " T " in l and l.split()[-1].startswith("fa_")))
    assert exported == declared_functions()


def test_binding_signatures_cover_the_header():
    import exact_tiled_attention_10_gb300 as fa
    assert set(declared_functions()) == set(fa._SIGS)


def test_params_struct_matches_the_header():
    """The ctypes mirror has the C struct's fields in the C order."""
    import exact_tiled_attention_10_gb300 as fa
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct \{(.*?)\} fa_attn_params;", src, flags=re.S).group(1)
    names = []
    for decl in body.split(";"):
        decl = decl.strip()
        if not decl:
            continue
        parts = [x.strip() for x in decl.split(",")]
        first = parts[0].split()[-1].lstrip("*")
        names += [first] + [x.lstrip("*") for x in parts[1:]]
    assert names == [f[0] for f in fa.AttnParams._fields_]
    p = fa.attn_params()
    assert p.struct_size == ctypes.sizeof(fa.AttnParams)
    assert (p.window_left, p.window_right, p.num_splits, p.dtype, p.layout) == (-1, -1, 1, 0, 0)


def test_version_and_sizes(lib):
    lib.fa_version.restype = ctypes.c_int
    assert lib.fa_version() >= 1
    lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fa_bwd_workspace_size.argtypes = [ctypes.c_int] * 4
    # bf16: lse2 + D (B*H*Np floats each) + dQ accumulator (B*H*Np*d floats), Np = 384
    B, H, N, d = 2, 3, 300, 128
    Np = 384
    expect = 2 * (B * H * Np * 4) + B * H * Np * d * 4
    assert lib.fa_bwd_workspace_size(B, H, N, d) == expect
    assert lib.fa_bwd_workspace_size(B, H, N, 96) == 0
    lib.fa_fp8_num_blocks.restype = ctypes.c_int
    assert lib.fa_fp8_num_blocks(16384) == 256 and lib.fa_fp8_num_blocks(65) == 2


def test_split_plan_without_gpu():
    """Split-key plan (fa_attn_fwd_splits / fa_attn_fwd_workspace_size) for a
    152-SM device (the default when no GPU is visible).  Long_head (B=2 H=16
    N=4096) and long_seq (B=1 H=8 N=16384) both have 512 items of 256 query
    rows: 3 full rounds of 152 plus 56; splitting those 56 into 2 key ranges
    makes the last round half as long (estimated 120 vs 136 key blocks, resp.
    456 vs 520), so 56 * 2 = 112 partials of 256 rows x (128 + 1) float32."""
    import exact_tiled_attention_10_gb300 as fa
    cnt, wsz = fa.split_count, fa.split_workspace_size
    expect = 112 * 256 * 128 * 4 + 112 * 256 * 4
    assert cnt(2, 16, 4096, 128) == 2 and wsz(2, 16, 4096, 128) == expect
    assert cnt(1, 8, 16384, 128) == 2 and wsz(1, 8, 16384, 128) == expect
    # causal and key-padded calls are not split automatically; num_splits=1 never
    assert cnt(2, 16, 4096, 128, causal=True) == 1 and wsz(2, 16, 4096, 128, causal=True) == 0
    assert cnt(2, 16, 4096, 128, kv_lens=True) == 1
    assert cnt(2, 16, 4096, 128, num_splits=1) == 1
    # explicit splits: every item, capped at 64
    assert cnt(2, 2, 300, 64, causal=True, num_splits=3) == 3
    assert wsz(2, 2, 300, 64, causal=True, num_splits=3) == (2 * 2 * 2) * 3 * 256 * (64 + 1) * 4
    assert cnt(2, 2, 300, 64, num_splits=1000) == 64


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


def _status(bwd=False, **fields):
    import exact_tiled_attention_10_gb300 as fa
    lib = fa.load_library()
    p = fa.attn_params(**fields)
    return (lib.fa_attn_bwd if bwd else lib.fa_attn_fwd)(ctypes.byref(p), None)


def _ws(bwd=False, **fields):
    import exact_tiled_attention_10_gb300 as fa
    lib = fa.load_library()
    p = fa.attn_params(**fields)
    return int((lib.fa_attn_bwd_workspace_size if bwd else lib.fa_attn_fwd_workspace_size)(ctypes.byref(p)))


A = 4096  # a 16-byte aligned fake device address: every case below is refused before any use
FWD = dict(q=A, k=A, v=A, o=A, lse=A)
BWD = dict(FWD, dout=A, dq=A, dk=A, dv=A)


def test_one_validation_routine_refuses_the_combinations_not_built():
    """fa_attn_fwd / fa_attn_bwd refuse, on the host and before any CUDA
    call, every combination the library does not build (FA_ERR_UNSUPPORTED),
    and malformed parameter blocks (FA_ERR_INVALID_ARG).  (The d = 64 FP8
    case runs the host checks up to the head dimension, which comes before
    any CUDA call.)"""
    import exact_tiled_attention_10_gb300 as fa
    base = dict(batch=2, heads=4, seqlen_q=256, head_dim=128, scale=0.1)
    U, I = fa.FA_ERR_UNSUPPORTED, fa.FA_ERR_INVALID_ARG
    # FP8: packed / [B,N,H,d] layouts, windows, block lists, N_q != N_k, a backward
    assert _status(**base, **FWD, dtype=fa.FA_E4M3, layout=fa.FA_LAYOUT_BNHD) == U
    assert _status(**base, **FWD, dtype=fa.FA_E4M3, window_left=64) == U
    assert _status(**base, **FWD, dtype=fa.FA_E4M3, block_row_ptr=A, block_col_idx=A) == U
    assert _status(**base, **FWD, dtype=fa.FA_E4M3, seqlen_k=300) == U
    assert _status(True, **base, **BWD, dtype=fa.FA_E4M3, kv_heads=2) == U
    assert _status(True, **base, **BWD, dtype=fa.FA_E4M3, deterministic=1) == U
    assert _status(True, **dict(base, head_dim=64), **BWD, dtype=fa.FA_E4M3, q_scale=A, k_scale=A, v_scale=A, workspace=A,
                   workspace_bytes=1 << 30) == U
    assert _status(**base, **FWD, dtype=fa.FA_E4M3, kv_heads=2, num_splits=0) == U
    # float32: anything beyond causal, kv_lens and block_c
    assert _status(**base, **FWD, dtype=fa.FA_F32, window_right=0) == U
    assert _status(**base, **FWD, dtype=fa.FA_F32, kv_heads=2) == U
    assert _status(True, **base, **BWD, dtype=fa.FA_F32, deterministic=1) == U
    # packed sequences: separate key ranges with a window; kv_lens; splits
    packed = dict(base, layout=fa.FA_LAYOUT_PACKED, total_q=512, cu_seqlens_q=A)
    assert _status(**packed, **FWD, cu_seqlens_k=A, window_left=5) == U
    assert _status(**packed, **FWD, kv_lens=A) == U
    assert _status(**packed, **FWD, num_splits=0) == U
    assert _status(**dict(packed, cu_seqlens_q=None), **FWD) == I
    # [B, N, H, d]: key lengths, windows
    assert _status(**base, **FWD, layout=fa.FA_LAYOUT_BNHD, kv_lens=A) == U
    assert _status(**base, **FWD, layout=fa.FA_LAYOUT_BNHD, window_left=3) == U
    # N_q != N_k with a window or block lists; block lists with a window
    assert _status(**base, **FWD, seqlen_k=1000, window_left=3) == U
    assert _status(**base, **FWD, seqlen_k=1000, block_row_ptr=A, block_col_idx=A) == U
    assert _status(**base, **FWD, window_left=3, block_row_ptr=A, block_col_idx=A) == U
    # options of the other pass
    assert _status(True, **base, **BWD, num_splits=2) == U
    assert _status(**base, **FWD, deterministic=1) == U
    # malformed blocks
    assert _status(**base, **FWD, window_left=-2) == I
    assert _status(**base, **FWD, kv_heads=3) == I
    assert _status(**base, **FWD, block_row_ptr=A) == I
    assert _status(**base, **FWD, dtype=7) == I
    assert _status(**base, **FWD, layout=9) == I
    assert _status(**dict(base, batch=0), **FWD) == I
    import exact_tiled_attention_10_gb300 as fa2
    p = fa2.attn_params(**base, **FWD)
    p.struct_size = 8
    assert fa2.load_library().fa_attn_fwd(ctypes.byref(p), None) == I
    assert b"struct_size" in fa2.load_library().fa_last_error()


def test_host_validation_of_the_variant_paths():
    """Bad arguments of the window, block-sparse, rectangular, grouped and
    fused-quantiser paths are refused on the host, before any CUDA call (so
    this runs without a GPU)."""
    import exact_tiled_attention_10_gb300 as fa
    lib = fa.load_library()
    I, U = fa.FA_ERR_INVALID_ARG, fa.FA_ERR_UNSUPPORTED
    # [B, N, H, d] layout: unsupported head dim, B * N beyond 32 bits, workspace too small
    bnhd = dict(layout=fa.FA_LAYOUT_BNHD, batch=2, heads=4, seqlen_q=256, head_dim=128, scale=0.1)
    assert _status(**dict(bnhd, head_dim=96), **FWD) == U
    assert _status(**dict(bnhd, batch=1 << 16, seqlen_q=1 << 16), **FWD) == I
    assert _ws(True, **bnhd) == _ws(True, **dict(bnhd, layout=fa.FA_LAYOUT_PACKED, total_q=512, cu_seqlens_q=A)) > 0
    assert _status(True, **bnhd, **BWD, workspace=A, workspace_bytes=1024) == I
    # packed sliding window: a bad edge; separate key ranges need more workspace when deterministic
    packed = dict(layout=fa.FA_LAYOUT_PACKED, batch=2, heads=4, seqlen_q=256, total_q=512, head_dim=128,
                  scale=0.1, cu_seqlens_q=A)
    assert _status(**packed, **FWD, window_left=-2) == I
    kvr = dict(packed, kv_heads=2, seqlen_k=300, total_k=600, cu_seqlens_k=A)
    assert _ws(True, **dict(kvr, deterministic=1)) > _ws(True, **kvr) > 0
    # deterministic packed / [B, N, H, d]: more workspace than the default
    assert _ws(True, **dict(packed, batch=3, seqlen_q=300, heads=8, kv_heads=2, deterministic=1)) > \
        _ws(True, **dict(packed, batch=3, seqlen_q=300, heads=8, kv_heads=2))
    assert _status(True, **dict(packed, cu_seqlens_q=None), **BWD, deterministic=1, workspace=A,
                   workspace_bytes=1 << 30) == I
    # block-sparse: the transposed lists need workspace beyond the plain backward's
    sp = dict(batch=1, heads=4, seqlen_q=256, head_dim=128, scale=0.1, block_row_ptr=A, block_col_idx=A)
    need = _ws(True, **sp)
    assert need > lib.fa_bwd_workspace_size(1, 4, 256, 128)
    assert _status(True, **sp, **BWD, workspace=A, workspace_bytes=need - 1) == I
    # rectangular: negative split count; a decode step (one query per head, long
    # cache) is split, a long prefill is not
    assert _status(**dict(batch=1, heads=4, seqlen_q=1, seqlen_k=100, head_dim=128, scale=0.1), **FWD,
                   num_splits=-1) == I
    assert fa.rect_split_count(1, 32, 8, 1, 131072, 128, 0) > 1
    assert fa.rect_split_count(8, 32, 8, 4096, 4096, 128, 0) == 1
    # fused quantiser: bad group
    assert lib.fa_quantize_fp8_qkv(A, A, A, A, A, A, A, A, A, 1, 4, 3, 256, 128, None) == 1
    # grouped backward: the split workspace is larger only when key blocks are few
    g = dict(batch=2, heads=16, kv_heads=2, seqlen_q=4096, head_dim=128, scale=0.1)
    assert _ws(True, **g) > lib.fa_bwd_workspace_size(2, 16, 4096, 128)
    g2 = dict(g, batch=64, kv_heads=16)
    assert _ws(True, **g2) <= lib.fa_bwd_workspace_size(64, 16, 4096, 128) + 256


def test_deterministic_backward_workspace_without_gpu():
    """The deterministic backward's workspace: fa_bwd's layout, then A - 1
    more float32 dQ accumulators and A x 4 turn counters per dQ tile, where
    A = min(8, key blocks, ceil(152 / (B * Hkv)) + 1) depends on the shape
    only; argument errors are caught on the host."""
    import exact_tiled_attention_10_gb300 as fa
    lib = fa.load_library()
    for (B, H, Hkv, N, d) in [(2, 16, 16, 4096, 128), (1, 8, 1, 300, 64), (64, 16, 16, 1024, 128)]:
        Np = -(-N // 128) * 128
        kt = -(-N // 128)
        A_ = min(8, kt, -(-152 // (B * Hkv)) + 1)
        acc = B * H * Np * d * 4
        turns = A_ * B * H * (Np // (64 if d == 128 else 128)) * 4 * 4
        size = _ws(True, batch=B, heads=H, kv_heads=Hkv, seqlen_q=N, head_dim=d, scale=0.1, deterministic=1)
        assert size == lib.fa_bwd_workspace_size(B, H, N, d) + (A_ - 1) * acc + turns
    base = dict(batch=1, heads=4, seqlen_q=256, head_dim=128, scale=0.1, deterministic=1)
    assert _ws(True, **dict(base, kv_heads=3)) == 0 and _ws(True, **dict(base, head_dim=96)) == 0
    need = _ws(True, **base)
    # workspace below fa_bwd's own layout
    assert _status(True, **base, **BWD, workspace=A, workspace_bytes=1024) == fa.FA_ERR_INVALID_ARG
    assert need > 1024
