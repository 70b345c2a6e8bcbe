"""Exact tiled attention for GB300 (sm_103a): thin Python binding.

Every step of the computation runs in the CUDA kernels of ``libfa_gb300.so``
behind the C ABI of ``include/fa.h``; this module only marshals arguments
(torch tensors -> device pointers, the current CUDA stream) and allocates
outputs and scratch with torch.  There is no CPU fallback: if the library is
missing or no CUDA device is present, calls raise.

    o, lse = forward(q, k, v, causal=True)               # bf16 or float32
    dq, dk, dv = backward(q, k, v, o, lse, do, causal=True)
    q8, sq = quantize_fp8(q)                              # E4M3 + per-64-row scales
    o8, lse8 = forward_fp8(q8, k8, v8, sq, sk, sv)
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Tuple

import torch

__all__ = ["forward", "forward_split", "forward_varlen", "backward_varlen", "backward",
           "block_lists", "forward_block_sparse", "backward_block_sparse", "quantize_fp8_qkv", "forward_rect", "backward_rect", "quantize_fp8", "forward_fp8", "forward_fp8_split",
           "split_count", "split_workspace_size", "check_device_status",
           "selftest_wait_timeout",
           "bwd_workspace_size", "fwd_workspace_size", "library_path", "load_library", "FAError"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libfa_gb300.so")
_lock = threading.Lock()
_lib = None

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = 0, 1, 2, 3, 4
FA_BF16, FA_F32 = 0, 1
_STATUS = {1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_CUDA", 4: "FA_ERR_TIMEOUT"}

# C signatures of include/fa.h, as ctypes argtypes
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "fa_version": ([], _i),
    "fa_last_error": ([], ctypes.c_char_p),
    "fa_check_device_status": ([_vp], _i),
    "fa_selftest_wait_timeout": ([ctypes.c_uint, _vp, _vp], _i),
    "fa_fwd": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _vp], _i),
    "fa_fwd_workspace_size": ([_i, _i, _i, _i, _i], _sz),
    "fa_fwd_ex": ([_i, _i, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _vp, _sz, _vp], _i),
    "fa_bwd_workspace_size": ([_i, _i, _i, _i, _i], _sz),
    "fa_bwd": ([_vp] * 9 + [_i, _i, _i, _i, _f, _i, _vp, _vp, _sz, _vp], _i),
    "fa_bwd_ex": ([_i] + [_vp] * 9 + [_i, _i, _i, _i, _f, _i, _vp, _vp, _sz, _vp], _i),
    "fa_bwd_preprocess": ([_vp, _vp, _vp, _i, _i, _i, _i, _vp, _sz, _vp], _i),
    "fa_bwd_main": ([_vp] * 6 + [_i, _i, _i, _i, _f, _i, _vp, _vp, _sz, _vp], _i),
    "fa_bwd_dq": ([_vp, _i, _i, _i, _i, _f, _vp, _sz, _vp], _i),
    "fa_bwd_noalloc_max_scratch": ([], _sz),
    "fa_bwd_noalloc": ([_vp] * 9 + [_i, _i, _i, _i, _f, _i, _vp, _vp], _i),
    "fa_fp8_num_blocks": ([_i], _i),
    "fa_quantize_fp8": ([_vp, _vp, _vp, _i, _i, _i, _i, _vp], _i),
    "fa_fwd_fp8": ([_vp] * 8 + [_i, _i, _i, _i, _f, _i, _vp, _vp], _i),
    "fa_fwd_gqa": ([_vp] * 5 + [_i, _i, _i, _i, _i, _f, _i, _vp, _vp], _i),
    "fa_fwd_window": ([_vp] * 5 + [_i, _i, _i, _i, _i, _f, _i, _i, _i, _vp, _vp], _i),
    "fa_bwd_window": ([_vp] * 9 + [_i, _i, _i, _i, _i, _f, _i, _i, _i, _vp, _vp, _sz, _vp], _i),
    "fa_fwd_block_sparse": ([_vp] * 5 + [_i, _i, _i, _i, _i, _f, _i, _vp, _vp, _vp, _vp], _i),
    "fa_bwd_block_sparse_workspace_size": ([_i] * 4, _sz),
    "fa_bwd_gqa_workspace_size": ([_i] * 5, _sz),
    "fa_bwd_deterministic_workspace_size": ([_i] * 5, _sz),
    "fa_bwd_deterministic": ([_vp] * 9 + [_i, _i, _i, _i, _i, _f, _i, _vp, _vp, _sz, _vp], _i),
    "fa_selftest_quantiser_division": ([_vp, _vp, _i, _sz, _vp, _vp, _vp], _i),
    "fa_quantize_fp8_qkv": ([_vp] * 9 + [_i] * 5 + [_vp], _i),
    "fa_fwd_rect_workspace_size": ([_i] * 7, _sz),
    "fa_fwd_rect_split_count": ([_i] * 7, _i),
    "fa_fwd_rect": ([_vp] * 5 + [_i] * 6 + [_f, _i, _vp, _i, _vp, _sz, _vp], _i),
    "fa_bwd_rect_workspace_size": ([_i] * 6, _sz),
    "fa_bwd_rect": ([_vp] * 9 + [_i] * 6 + [_f, _i, _vp, _vp, _sz, _vp], _i),
    "fa_bwd_block_sparse": ([_vp] * 9 + [_i, _i, _i, _i, _i, _f, _i, _vp, _vp, _vp, _vp, _sz, _vp], _i),
    "fa_fwd_varlen": ([_vp] * 6 + [_i, _i, _i, _i, _i, _i, _f, _i, _vp], _i),
    "fa_bwd_varlen_workspace_size": ([_i] * 4, _sz),
    "fa_bwd_varlen": ([_vp] * 10 + [_i, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp], _i),
    "fa_fwd_bnhd": ([_vp] * 5 + [_i, _i, _i, _i, _i, _f, _i, _vp], _i),
    "fa_fwd_varlen_kv": ([_vp] * 7 + [_i] * 7 + [_f, _i, _vp], _i),
    "fa_fwd_fp8_gqa": ([_vp] * 8 + [_i] * 5 + [_f, _i, _vp, _vp], _i),
    "fa_fwd_varlen_window": ([_vp] * 6 + [_i] * 6 + [_f, _i, _i, _i, _vp], _i),
    "fa_bwd_varlen_window": ([_vp] * 10 + [_i] * 6 + [_f, _i, _i, _i, _i, _vp, _sz, _vp], _i),
    "fa_bwd_varlen_kv_workspace_size": ([_i] * 7, _sz),
    "fa_bwd_varlen_kv": ([_vp] * 11 + [_i] * 8 + [_f, _i, _i, _vp, _sz, _vp], _i),
    "fa_bwd_bnhd_workspace_size": ([_i] * 4, _sz),
    "fa_bwd_bnhd": ([_vp] * 9 + [_i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp], _i),
    "fa_bwd_varlen_deterministic_workspace_size": ([_i] * 5, _sz),
    "fa_bwd_varlen_deterministic": ([_vp] * 10 + [_i, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp], _i),
    "fa_bwd_bnhd_deterministic_workspace_size": ([_i] * 5, _sz),
    "fa_bwd_bnhd_deterministic": ([_vp] * 9 + [_i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp], _i),
    "fa_bwd_window_deterministic": ([_vp] * 9 + [_i, _i, _i, _i, _i, _f, _i, _i, _i, _vp, _vp, _sz, _vp], _i),
    "fa_bwd_rect_deterministic_workspace_size": ([_i] * 6, _sz),
    "fa_bwd_block_sparse_deterministic_workspace_size": ([_i] * 5, _sz),
    "fa_bwd_block_sparse_deterministic": ([_vp] * 9 + [_i] * 5 + [_f, _i, _vp, _vp, _vp, _vp, _sz, _vp], _i),
    "fa_bwd_rect_deterministic": ([_vp] * 9 + [_i] * 6 + [_f, _i, _vp, _vp, _sz, _vp], _i),
    "fa_bwd_gqa": ([_vp] * 9 + [_i, _i, _i, _i, _i, _f, _i, _vp, _vp, _sz, _vp], _i),
    "fa_fwd_split_workspace_size": ([_i] * 7, _sz),
    "fa_fwd_split_count": ([_i] * 7, _i),
    "fa_fwd_split": ([_vp] * 5 + [_i, _i, _i, _i, _f, _i, _vp, _i, _vp, _sz, _vp], _i),
    "fa_fwd_fp8_split": ([_vp] * 8 + [_i, _i, _i, _i, _f, _i, _vp, _i, _vp, _sz, _vp], _i),
}


class FAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("%s: %s" % (_STATUS.get(status, str(status)), msg))
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libfa_gb300.so (built by ``build.build()``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    "libfa_gb300.so is not built; run exact_tiled_attention_10_gb300.build.build() "
                    "(the CUDA path has no fallback)")
            lib = ctypes.CDLL(_LIB_PATH)
            for name, (args, res) in _SIGS.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def _check(status: int):
    if status != FA_OK:
        raise FAError(status, load_library().fa_last_error().decode(errors="replace"))


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _need_cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("tensors must be on a CUDA device (no CPU fallback)")
            if not t.is_contiguous():
                raise ValueError("tensors must be contiguous")


def _kv(kv_lens: Optional[torch.Tensor], B: int, device) -> Optional[torch.Tensor]:
    if kv_lens is None:
        return None
    kv = kv_lens.to(device=device, dtype=torch.int32).contiguous()
    if kv.shape != (B,):
        raise ValueError("kv_lens must have shape [B]")
    return kv


def fwd_workspace_size(dtype: torch.dtype, B: int, H: int, N: int, d: int) -> int:
    dt = FA_F32 if dtype == torch.float32 else FA_BF16
    return int(load_library().fa_fwd_workspace_size(dt, B, H, N, d))


def bwd_workspace_size(dtype: torch.dtype, B: int, H: int, N: int, d: int) -> int:
    dt = FA_F32 if dtype == torch.float32 else FA_BF16
    return int(load_library().fa_bwd_workspace_size(dt, B, H, N, d))


def _window(window) -> Tuple[int, int]:
    if window is None:
        return -1, -1
    wl, wr = window
    wl = -1 if wl is None else int(wl)
    wr = -1 if wr is None else int(wr)
    if wl < -1 or wr < -1:
        raise ValueError("window edges must be >= -1 (-1 = unbounded)")
    return wl, wr


def forward(q, k, v, causal: bool = False, scale: Optional[float] = None, kv_lens=None,
            block_c: int = 0, out: Optional[torch.Tensor] = None,
            lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
            window: Optional[Tuple[int, int]] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """O, LSE of softmax(scale Q K^T + mask) V.  q: [B,H,N,d] bf16 or float32;
    k, v: [B,H,N,d], or bf16 [B,Hkv,N,d] with fewer key/value heads (H a
    multiple of Hkv; query head h uses key/value head h // (H // Hkv)).
    window = (left, right): sliding window, key j visible to query i only if
    i - left <= j <= i + right (-1 = unbounded; bf16 only)."""
    lib = load_library()
    _need_cuda(q, k, v)
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if (k.shape != (B, Hkv, N, d) or v.shape != k.shape or k.dtype != q.dtype or v.dtype != q.dtype
            or H % Hkv != 0):
        raise ValueError("q [B,H,N,d]; k, v [B,Hkv,N,d] with H a multiple of Hkv; one dtype")
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("dtype must be bfloat16 or float32")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q.device)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _need_cuda(o, l)
    wl, wr = _window(window)
    if wl >= 0 or wr >= 0:
        if q.dtype != torch.bfloat16:
            raise ValueError("the sliding window needs bfloat16 tensors")
        _check(lib.fa_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, H, Hkv, N, d, scale,
                                 int(bool(causal)), wl, wr, _ptr(kv), _stream(q)))
        return o, l
    if Hkv != H:
        if q.dtype != torch.bfloat16:
            raise ValueError("shared key/value heads need bfloat16 tensors")
        _check(lib.fa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, H, Hkv, N, d, scale,
                              int(bool(causal)), _ptr(kv), _stream(q)))
        return o, l
    dt = FA_F32 if q.dtype == torch.float32 else FA_BF16
    wsz = int(lib.fa_fwd_workspace_size(dt, B, H, N, d))
    ws = workspace
    if wsz and (ws is None or ws.numel() * ws.element_size() < wsz):
        ws = torch.empty(wsz, dtype=torch.uint8, device=q.device)
    _check(lib.fa_fwd_ex(dt, int(block_c), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, H, N, d,
                         scale, int(bool(causal)), _ptr(kv), _ptr(ws) if wsz else None, wsz,
                         _stream(q)))
    return o, l


def split_count(B: int, H: int, N: int, d: int, causal: bool = False, kv_lens: bool = False,
                num_splits: int = 0) -> int:
    """Number of key ranges fa_fwd_split uses for this call (1 = not split)."""
    return int(load_library().fa_fwd_split_count(B, H, N, d, int(bool(causal)), int(bool(kv_lens)),
                                                 int(num_splits)))


def split_workspace_size(B: int, H: int, N: int, d: int, causal: bool = False, kv_lens: bool = False,
                         num_splits: int = 0) -> int:
    return int(load_library().fa_fwd_split_workspace_size(B, H, N, d, int(bool(causal)), int(bool(kv_lens)),
                                                          int(num_splits)))


def _split_ws(B, H, N, d, causal, kv, num_splits, workspace, device):
    wsz = split_workspace_size(B, H, N, d, causal, kv is not None, num_splits)
    ws = workspace
    if wsz and (ws is None or ws.numel() * ws.element_size() < wsz):
        ws = torch.empty(wsz, dtype=torch.uint8, device=device)
    return (_ptr(ws) if wsz else None), wsz


def forward_split(q, k, v, causal: bool = False, scale: Optional[float] = None, kv_lens=None,
                  num_splits: int = 0, out: Optional[torch.Tensor] = None,
                  lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None
                  ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Split-key bf16 forward (FlashDecoding form): as forward(), with the key
    sequence of each query block cut into ranges merged by a second kernel.
    num_splits 0 = automatic, 1 = none, >= 2 = that many ranges per item."""
    lib = load_library()
    _need_cuda(q, k, v)
    B, H, N, d = q.shape
    if q.dtype != torch.bfloat16 or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("forward_split takes bfloat16 q, k, v")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q.device)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    wsp, wsz = _split_ws(B, H, N, d, causal, kv, num_splits, workspace, q.device)
    _check(lib.fa_fwd_split(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, H, N, d, scale,
                            int(bool(causal)), _ptr(kv), int(num_splits), wsp, wsz, _stream(q)))
    return o, l


def block_lists(block_mask, device) -> Tuple[torch.Tensor, torch.Tensor]:
    """(row_ptr, col_idx) int32 device tensors of a 0/1 block mask
    [nb][nb] (query block x key block, 128 x 128 blocks)."""
    bm = torch.as_tensor(block_mask).to("cpu").bool()
    if bm.dim() != 2 or bm.shape[0] != bm.shape[1]:
        raise ValueError("block_mask must be a square [nb, nb] matrix")
    counts = bm.sum(dim=1).to(torch.int32)
    row_ptr = torch.zeros(bm.shape[0] + 1, dtype=torch.int32)
    row_ptr[1:] = torch.cumsum(counts, 0)
    col_idx = bm.nonzero()[:, 1].to(torch.int32)  # row-major: ascending within each row
    return row_ptr.to(device), col_idx.to(device)


def forward_block_sparse(q, k, v, row_ptr, col_idx, causal: bool = False, scale: Optional[float] = None,
                         kv_lens=None, out: Optional[torch.Tensor] = None,
                         lse: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Block-sparse forward (128 x 128 blocks): query block i attends to the
    key blocks col_idx[row_ptr[i]:row_ptr[i+1]] only (see block_lists)."""
    lib = load_library()
    _need_cuda(q, k, v, row_ptr, col_idx)
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if q.dtype != torch.bfloat16 or k.shape != (B, Hkv, N, d) or v.shape != k.shape or H % Hkv != 0:
        raise ValueError("q [B,H,N,d]; k, v [B,Hkv,N,d] bfloat16 with H a multiple of Hkv")
    if row_ptr.dtype != torch.int32 or col_idx.dtype != torch.int32 or row_ptr.numel() != (N + 127) // 128 + 1:
        raise ValueError("row_ptr int32 [ceil(N/128) + 1], col_idx int32")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q.device)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(lib.fa_fwd_block_sparse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, H, Hkv, N, d, scale,
                                   int(bool(causal)), _ptr(row_ptr), _ptr(col_idx), _ptr(kv), _stream(q)))
    return o, l


def backward_block_sparse(q, k, v, o, lse, dout, row_ptr, col_idx, causal: bool = False,
                          scale: Optional[float] = None, kv_lens=None, workspace: Optional[torch.Tensor] = None,
                          deterministic: bool = False):
    """Backward of forward_block_sparse: dQ [B,H,N,d], dK, dV [B,Hkv,N,d].
    deterministic: bitwise reproducible gradients (see backward)."""
    lib = load_library()
    _need_cuda(q, k, v, o, lse, dout, row_ptr, col_idx)
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q.device)
    wsz = int(lib.fa_bwd_block_sparse_deterministic_workspace_size(B, H, Hkv, N, d) if deterministic
              else lib.fa_bwd_block_sparse_workspace_size(B, H, N, d))
    ws = workspace
    if ws is None or ws.numel() * ws.element_size() < wsz:
        ws = torch.empty(wsz, dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fn = lib.fa_bwd_block_sparse_deterministic if deterministic else lib.fa_bwd_block_sparse
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
              _ptr(dv), B, H, Hkv, N, d, scale, int(bool(causal)), _ptr(row_ptr),
              _ptr(col_idx), _ptr(kv), _ptr(ws), ws.numel() * ws.element_size(),
              _stream(q)))
    return dq, dk, dv


def forward_rect(q, k, v, causal: bool = False, scale: Optional[float] = None, kv_lens=None,
                 num_splits: int = 0, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Nq queries against Nk keys (decoding against a key/value cache,
    cross-attention): q [B,H,Nq,d], k, v [B,Hkv,Nk,d] bf16.  Causal: the
    queries are the last Nq positions (query i sees keys j <= i + Nk - Nq)."""
    lib = load_library()
    _need_cuda(q, k, v)
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if (q.dtype != torch.bfloat16 or k.dtype != q.dtype or v.dtype != q.dtype or k.shape != (B, Hkv, Nk, d)
            or v.shape != k.shape or H % Hkv != 0):
        raise ValueError("q [B,H,Nq,d]; k, v [B,Hkv,Nk,d] bfloat16 with H a multiple of Hkv")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q.device)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    wsz = int(lib.fa_fwd_rect_workspace_size(B, H, Hkv, Nq, Nk, d, int(num_splits)))
    ws = workspace
    if wsz and (ws is None or ws.numel() * ws.element_size() < wsz):
        ws = torch.empty(wsz, dtype=torch.uint8, device=q.device)
    _check(lib.fa_fwd_rect(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, H, Hkv, Nq, Nk, d, scale,
                           int(bool(causal)), _ptr(kv), int(num_splits), _ptr(ws) if wsz else None, wsz,
                           _stream(q)))
    return o, l


def backward_rect(q, k, v, o, lse, dout, causal: bool = False, scale: Optional[float] = None, kv_lens=None,
                  workspace: Optional[torch.Tensor] = None, deterministic: bool = False):
    """Backward of forward_rect: dQ [B,H,Nq,d], dK, dV [B,Hkv,Nk,d].
    deterministic: bitwise reproducible gradients (see backward)."""
    lib = load_library()
    _need_cuda(q, k, v, o, lse, dout)
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q.device)
    wsz = int(lib.fa_bwd_rect_deterministic_workspace_size(B, H, Hkv, Nq, Nk, d) if deterministic
              else lib.fa_bwd_rect_workspace_size(B, H, Hkv, Nq, Nk, d))
    ws = workspace
    if ws is None or ws.numel() * ws.element_size() < wsz:
        ws = torch.empty(wsz, dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fn = lib.fa_bwd_rect_deterministic if deterministic else lib.fa_bwd_rect
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
              B, H, Hkv, Nq, Nk, d, scale, int(bool(causal)), _ptr(kv), _ptr(ws),
              ws.numel() * ws.element_size(), _stream(q)))
    return dq, dk, dv


def _cu(cu_seqlens, device):
    cu = cu_seqlens.to(device=device, dtype=torch.int32).contiguous()
    if cu.dim() != 1 or cu.numel() < 2:
        raise ValueError("cu_seqlens must be a 1-D tensor of batch + 1 offsets")
    return cu


def forward_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = False,
                   scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                   lse: Optional[torch.Tensor] = None, cu_seqlens_k=None,
                   window: Optional[Tuple[int, int]] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Packed variable-length forward: q [total, H, d], k, v [total, Hkv, d]
    (bf16), sequence b = tokens cu_seqlens[b] .. cu_seqlens[b+1]-1.  Returns
    O [total, H, d] and LSE [H, total].  cu_seqlens_k: the sequences' own key
    ranges in k, v [total_k, Hkv, d] (flash_attn_varlen_func's cu_seqlens_k;
    with causal, the queries are each sequence's last positions).  window:
    the sliding window (see forward), within each sequence."""
    lib = load_library()
    _need_cuda(q, k, v)
    T, H, d = q.shape
    Hkv = k.shape[1]
    Tk = k.shape[0]
    if (q.dtype != torch.bfloat16 or k.dtype != q.dtype or v.dtype != q.dtype or k.shape != (Tk, Hkv, d)
            or v.shape != k.shape or H % Hkv != 0 or (cu_seqlens_k is None and Tk != T)):
        raise ValueError("q [total,H,d], k, v [total(_k),Hkv,d] bfloat16 with H a multiple of Hkv")
    cu = _cu(cu_seqlens, q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((H, T), dtype=torch.float32, device=q.device) if lse is None else lse
    wl, wr = _window(window)
    if wl >= 0 or wr >= 0:
        _check(lib.fa_fwd_varlen_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), _ptr(cu), cu.numel() - 1, T,
                                        int(max_seqlen), H, Hkv, d, scale, int(bool(causal)), wl, wr, _stream(q)))
        return o, l
    if cu_seqlens_k is not None:
        cuk = _cu(cu_seqlens_k, q.device)
        _check(lib.fa_fwd_varlen_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), _ptr(cu), _ptr(cuk), cu.numel() - 1,
                                    T, Tk, int(max_seqlen), H, Hkv, d, scale, int(bool(causal)), _stream(q)))
        return o, l
    _check(lib.fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), _ptr(cu), cu.numel() - 1, T,
                             int(max_seqlen), H, Hkv, d, scale, int(bool(causal)), _stream(q)))
    return o, l


def _bnhd_shapes(q, k, v):
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    if (q.dtype != torch.bfloat16 or k.dtype != q.dtype or v.dtype != q.dtype or k.shape != (B, N, Hkv, d)
            or v.shape != k.shape or H % Hkv != 0):
        raise ValueError("q [B,N,H,d], k, v [B,N,Hkv,d] bfloat16 with H a multiple of Hkv")
    return B, N, H, Hkv, d


def forward_bnhd(q, k, v, causal: bool = False, scale: Optional[float] = None,
                 out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None):
    """Forward on flash_attn_func's layout: q [B,N,H,d], k, v [B,N,Hkv,d]
    (bf16).  Returns O [B,N,H,d] and LSE [B,H,N] (float32)."""
    lib = load_library()
    _need_cuda(q, k, v)
    B, N, H, Hkv, d = _bnhd_shapes(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(lib.fa_fwd_bnhd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, N, H, Hkv, d, scale,
                           int(bool(causal)), _stream(q)))
    return o, l


def backward_bnhd(q, k, v, o, lse, dout, causal: bool = False, scale: Optional[float] = None,
                  workspace: Optional[torch.Tensor] = None, deterministic: bool = False):
    """dQ [B,N,H,d], dK, dV [B,N,Hkv,d] of forward_bnhd (dK, dV summed over
    the query heads sharing a key/value head).  deterministic: bitwise
    reproducible gradients (see backward)."""
    lib = load_library()
    _need_cuda(q, k, v, o, lse, dout)
    B, N, H, Hkv, d = _bnhd_shapes(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    wsz = int(lib.fa_bwd_bnhd_deterministic_workspace_size(B, N, H, Hkv, d) if deterministic
              else lib.fa_bwd_bnhd_workspace_size(B, N, H, d))
    ws = workspace
    if ws is None or ws.numel() * ws.element_size() < wsz:
        ws = torch.empty(wsz, dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fn = lib.fa_bwd_bnhd_deterministic if deterministic else lib.fa_bwd_bnhd
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
              _ptr(dv), B, N, H, Hkv, d, scale, int(bool(causal)), _ptr(ws),
              ws.numel() * ws.element_size(), _stream(q)))
    return dq, dk, dv


def backward_varlen(q, k, v, o, lse, dout, cu_seqlens, max_seqlen: int, causal: bool = False,
                    scale: Optional[float] = None, workspace: Optional[torch.Tensor] = None,
                    deterministic: bool = False, cu_seqlens_k=None, max_seqlen_k: Optional[int] = None,
                    window: Optional[Tuple[int, int]] = None):
    """Backward of forward_varlen: dQ [total, H, d], dK, dV [total(_k), Hkv, d].
    deterministic: bitwise reproducible gradients (see backward).
    cu_seqlens_k / max_seqlen_k: separate key ranges (see forward_varlen)."""
    lib = load_library()
    _need_cuda(q, k, v, o, lse, dout)
    T, H, d = q.shape
    Hkv = k.shape[1]
    cu = _cu(cu_seqlens, q.device)
    batch = cu.numel() - 1
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    wl, wr = _window(window)
    if wl >= 0 or wr >= 0:
        wsz = int(lib.fa_bwd_varlen_deterministic_workspace_size(batch, int(max_seqlen), H, Hkv, d) if deterministic
                  else lib.fa_bwd_varlen_workspace_size(batch, int(max_seqlen), H, d))
        ws = workspace
        if ws is None or ws.numel() * ws.element_size() < wsz:
            ws = torch.empty(wsz, dtype=torch.uint8, device=q.device)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        _check(lib.fa_bwd_varlen_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                                        _ptr(dk), _ptr(dv), _ptr(cu), batch, T, int(max_seqlen), H, Hkv, d, scale,
                                        int(bool(causal)), wl, wr, int(bool(deterministic)), _ptr(ws),
                                        ws.numel() * ws.element_size(), _stream(q)))
        return dq, dk, dv
    if cu_seqlens_k is not None:
        cuk = _cu(cu_seqlens_k, q.device)
        mk = int(max_seqlen if max_seqlen_k is None else max_seqlen_k)
        wsz = int(lib.fa_bwd_varlen_kv_workspace_size(batch, int(max_seqlen), mk, H, Hkv, d, int(bool(deterministic))))
        ws = workspace
        if ws is None or ws.numel() * ws.element_size() < wsz:
            ws = torch.empty(wsz, dtype=torch.uint8, device=q.device)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        _check(lib.fa_bwd_varlen_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                    _ptr(dv), _ptr(cu), _ptr(cuk), batch, T, k.shape[0], int(max_seqlen), mk, H, Hkv,
                                    d, scale, int(bool(causal)), int(bool(deterministic)), _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(q)))
        return dq, dk, dv
    wsz = int(lib.fa_bwd_varlen_deterministic_workspace_size(batch, int(max_seqlen), H, Hkv, d) if deterministic
              else lib.fa_bwd_varlen_workspace_size(batch, int(max_seqlen), H, d))
    ws = workspace
    if ws is None or ws.numel() * ws.element_size() < wsz:
        ws = torch.empty(wsz, dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fn = lib.fa_bwd_varlen_deterministic if deterministic else lib.fa_bwd_varlen
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
              _ptr(dv), _ptr(cu), batch, T, int(max_seqlen), H, Hkv, d, scale,
              int(bool(causal)), _ptr(ws), ws.numel() * ws.element_size(), _stream(q)))
    return dq, dk, dv


def backward(q, k, v, o, lse, dout, causal: bool = False, scale: Optional[float] = None,
             kv_lens=None, workspace: Optional[torch.Tensor] = None,
             dq: Optional[torch.Tensor] = None, dk: Optional[torch.Tensor] = None,
             dv: Optional[torch.Tensor] = None, window: Optional[Tuple[int, int]] = None,
             deterministic: bool = False):
    """dQ, dK, dV of L = sum(O * dout).  With fewer key/value heads (k, v
    [B,Hkv,N,d]), dK and dV sum over the query heads sharing each one.
    window: the forward's sliding window (see forward).
    deterministic: bitwise-reproducible gradients (bf16, no window): the dQ
    parts are added in key-block order."""
    lib = load_library()
    _need_cuda(q, k, v, o, lse, dout)
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q.device)
    dt = FA_F32 if q.dtype == torch.float32 else FA_BF16
    wl, wr = _window(window)
    grouped = Hkv != H or wl >= 0 or wr >= 0
    if deterministic:
        if dt != FA_BF16 or H % Hkv != 0:
            raise ValueError("the deterministic backward takes bfloat16 tensors and H a multiple of Hkv")
        wsz = int(lib.fa_bwd_deterministic_workspace_size(B, H, Hkv, N, d))
    else:
        wsz = int(lib.fa_bwd_gqa_workspace_size(B, H, Hkv, N, d) if grouped and dt == FA_BF16
                  else lib.fa_bwd_workspace_size(dt, B, H, N, d))
    ws = workspace
    if ws is None or ws.numel() * ws.element_size() < wsz:
        ws = torch.empty(wsz, dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _need_cuda(dq, dk, dv)
    if deterministic and (wl >= 0 or wr >= 0):
        _check(lib.fa_bwd_window_deterministic(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                                               _ptr(dk), _ptr(dv), B, H, Hkv, N, d, scale, int(bool(causal)), wl, wr,
                                               _ptr(kv), _ptr(ws), ws.numel() * ws.element_size(), _stream(q)))
        return dq, dk, dv
    if deterministic:
        _check(lib.fa_bwd_deterministic(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                                        _ptr(dk), _ptr(dv), B, H, Hkv, N, d, scale, int(bool(causal)), _ptr(kv),
                                        _ptr(ws), ws.numel() * ws.element_size(), _stream(q)))
        return dq, dk, dv
    if wl >= 0 or wr >= 0:
        if q.dtype != torch.bfloat16 or H % Hkv != 0:
            raise ValueError("the sliding window needs bfloat16 tensors and H a multiple of Hkv")
        _check(lib.fa_bwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                                 _ptr(dk), _ptr(dv), B, H, Hkv, N, d, scale, int(bool(causal)), wl, wr,
                                 _ptr(kv), _ptr(ws), ws.numel() * ws.element_size(), _stream(q)))
        return dq, dk, dv
    if Hkv != H:
        if q.dtype != torch.bfloat16 or H % Hkv != 0:
            raise ValueError("shared key/value heads need bfloat16 tensors and H a multiple of Hkv")
        _check(lib.fa_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                              _ptr(dk), _ptr(dv), B, H, Hkv, N, d, scale, int(bool(causal)), _ptr(kv),
                              _ptr(ws), ws.numel() * ws.element_size(), _stream(q)))
        return dq, dk, dv
    _check(lib.fa_bwd_ex(dt, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                         _ptr(dk), _ptr(dv), B, H, N, d, scale, int(bool(causal)), _ptr(kv),
                         _ptr(ws), ws.numel() * ws.element_size(), _stream(q)))
    return dq, dk, dv


def quantize_fp8(x: torch.Tensor, out: Optional[torch.Tensor] = None,
                 scales: Optional[torch.Tensor] = None):
    """E4M3 codes (uint8 [B,H,N,d]) and float32 scales [B,H,ceil(N/64)] of a bf16 tensor."""
    lib = load_library()
    _need_cuda(x)
    if x.dtype != torch.bfloat16:
        raise ValueError("quantize_fp8 takes bfloat16 input")
    B, H, N, d = x.shape
    x8 = torch.empty(x.shape, dtype=torch.uint8, device=x.device) if out is None else out
    sc = torch.empty((B, H, lib.fa_fp8_num_blocks(N)), dtype=torch.float32, device=x.device) \
        if scales is None else scales
    _check(lib.fa_quantize_fp8(_ptr(x), _ptr(x8), _ptr(sc), B, H, N, d, _stream(x)))
    return x8, sc


def quantize_fp8_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor):
    """quantize_fp8 of q [B,H,N,d], k, v [B,Hkv,N,d] (bf16) in one launch:
    ((q8, sq), (k8, sk), (v8, sv))."""
    lib = load_library()
    _need_cuda(q, k, v)
    if q.dtype != torch.bfloat16 or k.dtype != q.dtype or v.dtype != q.dtype or k.shape != v.shape:
        raise ValueError("q [B,H,N,d], k, v [B,Hkv,N,d] bfloat16")
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    nb = lib.fa_fp8_num_blocks(N)
    out = []
    for t, h in ((q, H), (k, Hkv), (v, Hkv)):
        out.append((torch.empty(t.shape, dtype=torch.uint8, device=t.device),
                    torch.empty((B, h, nb), dtype=torch.float32, device=t.device)))
    _check(lib.fa_quantize_fp8_qkv(_ptr(q), _ptr(k), _ptr(v), _ptr(out[0][0]), _ptr(out[1][0]), _ptr(out[2][0]),
                                   _ptr(out[0][1]), _ptr(out[1][1]), _ptr(out[2][1]), B, H, Hkv, N, d, _stream(q)))
    return tuple(out)


def forward_fp8(q8, k8, v8, sq, sk, sv, causal: bool = False, scale: Optional[float] = None,
                kv_lens=None, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None):
    """FP8 E4M3 forward with per-64-row-block scales; O bf16, LSE float32.
    k8, v8 may have fewer heads (shared key/value heads)."""
    lib = load_library()
    _need_cuda(q8, k8, v8, sq, sk, sv)
    B, H, N, d = q8.shape
    Hkv = k8.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q8.device)
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q8.device) if lse is None else lse
    if Hkv != H:
        _check(lib.fa_fwd_fp8_gqa(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(sq), _ptr(sk), _ptr(sv), _ptr(o),
                                  _ptr(l), B, H, Hkv, N, d, scale, int(bool(causal)), _ptr(kv), _stream(q8)))
        return o, l
    _check(lib.fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(sq), _ptr(sk), _ptr(sv), _ptr(o),
                          _ptr(l), B, H, N, d, scale, int(bool(causal)), _ptr(kv), _stream(q8)))
    return o, l


def forward_fp8_split(q8, k8, v8, sq, sk, sv, causal: bool = False, scale: Optional[float] = None,
                      kv_lens=None, num_splits: int = 0, out: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None):
    """Split-key FP8 forward: forward_fp8 with the key ranges of forward_split."""
    lib = load_library()
    _need_cuda(q8, k8, v8, sq, sk, sv)
    B, H, N, d = q8.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q8.device)
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q8.device) if lse is None else lse
    wsp, wsz = _split_ws(B, H, N, d, causal, kv, num_splits, workspace, q8.device)
    _check(lib.fa_fwd_fp8_split(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(sq), _ptr(sk), _ptr(sv), _ptr(o),
                                _ptr(l), B, H, N, d, scale, int(bool(causal)), _ptr(kv), int(num_splits),
                                wsp, wsz, _stream(q8)))
    return o, l


def selftest_wait_timeout(limit_us: int = 20000, device=None) -> int:
    """Run the bounded-wait self-test kernel; returns the device flag (0 = the
    wait gave up as designed).  The error word it sets is reported by the next
    check_device_status()."""
    lib = load_library()
    dev = torch.device("cuda") if device is None else torch.device(device)
    flag = torch.full((4,), 7, dtype=torch.int32, device=dev)
    _check(lib.fa_selftest_wait_timeout(int(limit_us), flag.data_ptr(),
                                        torch.cuda.current_stream(dev).cuda_stream))
    return int(flag[0].item())


def check_device_status(device=None) -> None:
    """Synchronise the current stream and raise if a kernel recorded a timed-out wait."""
    lib = load_library()
    dev = torch.device("cuda") if device is None else torch.device(device)
    _check(lib.fa_check_device_status(torch.cuda.current_stream(dev).cuda_stream))
