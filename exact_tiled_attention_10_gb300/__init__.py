"""Exact tiled attention for GB300 (sm_103a): thin Python binding.

Every step of the computation runs in the CUDA kernels of ``libfa_gb300.so``
behind the C ABI of ``include/fa.h``; this module only marshals arguments
(torch tensors -> device pointers, the current CUDA stream) and allocates
outputs and scratch with torch.  There is no CPU fallback: if the library is
missing or no CUDA device is present, calls raise.  With FA_DEBUG=1 in the
environment the checked build ``libfa_gb300_debug.so`` (``build(debug=True)``)
is loaded instead; a broken access rule then surfaces as FA_ERR_CHECK from
``check_device_status()``.

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

__all__ = ["forward", "forward_split", "forward_varlen", "backward_varlen", "backward", "forward_bnhd",
           "backward_bnhd", "block_lists", "forward_block_sparse", "backward_block_sparse", "quantize_fp8_qkv",
           "forward_rect", "backward_rect", "rect_split_count", "quantize_fp8", "forward_fp8", "forward_fp8_split",
           "backward_fp8",
           "split_count", "split_workspace_size", "check_device_status", "selftest_wait_timeout", "attn_params",
           "AttnParams", "bwd_workspace_size", "fwd_workspace_size", "library_path", "load_library", "FAError"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libfa_gb300_debug.so" if os.environ.get("FA_DEBUG") == "1" else "libfa_gb300.so")
_lock = threading.Lock()
_lib = None

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT, FA_ERR_CHECK = 0, 1, 2, 3, 4, 5
FA_BF16, FA_F32, FA_E4M3 = 0, 1, 2
FA_LAYOUT_BHND, FA_LAYOUT_BNHD, FA_LAYOUT_PACKED = 0, 1, 2
_STATUS = {1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_CUDA", 4: "FA_ERR_TIMEOUT", 5: "FA_ERR_CHECK"}


class AttnParams(ctypes.Structure):
    """ctypes mirror of fa_attn_params (include/fa.h), field for field."""
    _fields_ = [
        ("struct_size", ctypes.c_size_t),
        ("dtype", ctypes.c_int), ("layout", ctypes.c_int),
        ("batch", ctypes.c_int), ("heads", ctypes.c_int), ("kv_heads", ctypes.c_int),
        ("seqlen_q", ctypes.c_int), ("seqlen_k", ctypes.c_int), ("head_dim", ctypes.c_int),
        ("total_q", ctypes.c_int), ("total_k", ctypes.c_int),
        ("scale", ctypes.c_float),
        ("causal", ctypes.c_int),
        ("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
        ("num_splits", ctypes.c_int), ("block_c", ctypes.c_int), ("deterministic", ctypes.c_int),
        ("kv_lens", ctypes.c_void_p),
        ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
        ("block_row_ptr", ctypes.c_void_p), ("block_col_idx", ctypes.c_void_p),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("q_scale", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("dout", ctypes.c_void_p), ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
    ]


# C signatures of include/fa.h, as ctypes argtypes
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_pp = ctypes.POINTER(AttnParams)
_SIGS = {
    "fa_version": ([], _i),
    "fa_last_error": ([], ctypes.c_char_p),
    "fa_check_device_status": ([_vp], _i),
    "fa_selftest_wait_timeout": ([ctypes.c_uint, _vp, _vp], _i),
    "fa_selftest_quantiser_division": ([_vp, _vp, _i, _sz, _vp, _vp, _vp], _i),
    "fa_fwd": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _vp], _i),
    "fa_bwd_workspace_size": ([_i, _i, _i, _i], _sz),
    "fa_bwd": ([_vp] * 9 + [_i, _i, _i, _i, _f, _i, _vp, _vp, _sz, _vp], _i),
    "fa_fp8_num_blocks": ([_i], _i),
    "fa_quantize_fp8": ([_vp, _vp, _vp, _i, _i, _i, _i, _vp], _i),
    "fa_quantize_fp8_qkv": ([_vp] * 9 + [_i] * 5 + [_vp], _i),
    "fa_fwd_fp8": ([_vp] * 8 + [_i, _i, _i, _i, _f, _i, _vp, _vp], _i),
    "fa_attn_params_init": ([_pp], None),
    "fa_attn_fwd_workspace_size": ([_pp], _sz),
    "fa_attn_fwd_splits": ([_pp], _i),
    "fa_attn_bwd_workspace_size": ([_pp], _sz),
    "fa_attn_fwd": ([_pp, _vp], _i),
    "fa_attn_bwd": ([_pp, _vp], _i),
    "fa_bwd_preprocess": ([_vp, _vp, _vp, _i, _i, _i, _i, _vp, _sz, _vp], _i),
    "fa_bwd_main": ([_vp] * 6 + [_i, _i, _i, _i, _f, _i, _vp, _vp, _sz, _vp], _i),
    "fa_bwd_dq": ([_vp, _i, _i, _i, _i, _f, _vp, _sz, _vp], _i),
    "fa_bwd_noalloc_max_scratch": ([], _sz),
    "fa_bwd_noalloc": ([_vp] * 9 + [_i, _i, _i, _i, _f, _i, _vp, _vp], _i),
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
                    "%s is not built; run exact_tiled_attention_10_gb300.build.build(%s) "
                    "(the CUDA path has no fallback)" % (os.path.basename(_LIB_PATH),
                                                         "debug=True" if "debug" in _LIB_PATH else ""))
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


def attn_params(**fields) -> AttnParams:
    """An fa_attn_params block initialised by the library (defaults: bf16,
    [B,H,N,d], no window, no split), with `fields` set; tensors are passed as
    their device pointers."""
    lib = load_library()
    p = AttnParams()
    lib.fa_attn_params_init(ctypes.byref(p))
    for name, val in fields.items():
        if isinstance(val, torch.Tensor):
            val = val.data_ptr()
        setattr(p, name, val)
    return p


def _scratch(nbytes: int, device, given: Optional[torch.Tensor]) -> Optional[torch.Tensor]:
    if nbytes == 0:
        return None
    if given is not None and given.numel() * given.element_size() >= nbytes:
        return given
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def _run(p: AttnParams, t: torch.Tensor, bwd: bool, workspace: Optional[torch.Tensor] = None):
    """Size the workspace for p, then one fa_attn_fwd / fa_attn_bwd call."""
    lib = load_library()
    nbytes = int((lib.fa_attn_bwd_workspace_size if bwd else lib.fa_attn_fwd_workspace_size)(ctypes.byref(p)))
    ws = _scratch(nbytes, t.device, workspace)
    p.workspace = None if ws is None else ws.data_ptr()
    p.workspace_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check((lib.fa_attn_bwd if bwd else lib.fa_attn_fwd)(ctypes.byref(p), _stream(t)))


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float32:
        return FA_F32
    raise ValueError("dtype must be bfloat16 or float32")


def fwd_workspace_size(dtype: torch.dtype, B: int, H: int, N: int, d: int) -> int:
    """Scratch of the forward on [B,H,N,d] tensors of `dtype` (float32 only)."""
    p = attn_params(dtype=FA_F32 if dtype == torch.float32 else FA_BF16, batch=B, heads=H, seqlen_q=N,
                    head_dim=d, scale=1.0)
    return int(load_library().fa_attn_fwd_workspace_size(ctypes.byref(p)))


def bwd_workspace_size(dtype: torch.dtype, B: int, H: int, N: int, d: int) -> int:
    """Scratch of the backward on [B,H,N,d] tensors of `dtype`."""
    p = attn_params(dtype=FA_F32 if dtype == torch.float32 else FA_BF16, batch=B, heads=H, seqlen_q=N,
                    head_dim=d, scale=1.0)
    return int(load_library().fa_attn_bwd_workspace_size(ctypes.byref(p)))


def _window(window) -> Tuple[int, int]:
    if window is None:
        return -1, -1
    wl, wr = window
    wl = -1 if wl is None else int(wl)
    wr = -1 if wr is None else int(wr)
    if wl < -1 or wr < -1:
        raise ValueError("window edges must be >= -1 (-1 = unbounded)")
    return wl, wr


def _bhnd(q, k, v, name="q [B,H,N,d]; k, v [B,Hkv,N,d] with H a multiple of Hkv; one dtype"):
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if (k.shape != (B, Hkv, N, d) or v.shape != k.shape or k.dtype != q.dtype or v.dtype != q.dtype
            or H % Hkv != 0):
        raise ValueError(name)
    return B, H, Hkv, N, d


def forward(q, k, v, causal: bool = False, scale: Optional[float] = None, kv_lens=None,
            block_c: int = 0, out: Optional[torch.Tensor] = None,
            lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
            window: Optional[Tuple[int, int]] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """O, LSE of softmax(scale Q K^T + mask) V.  q: [B,H,N,d] bf16 or float32;
    k, v: [B,H,N,d], or bf16 [B,Hkv,N,d] with fewer key/value heads (H a
    multiple of Hkv; query head h uses key/value head h // (H // Hkv)).
    window = (left, right): sliding window, key j visible to query i only if
    i - left <= j <= i + right (-1 = unbounded; bf16 only)."""
    _need_cuda(q, k, v)
    B, H, Hkv, N, d = _bhnd(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q.device)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _need_cuda(o, l)
    wl, wr = _window(window)
    p = attn_params(dtype=_dtype(q), batch=B, heads=H, kv_heads=Hkv, seqlen_q=N, head_dim=d, scale=scale,
                    causal=int(bool(causal)), window_left=wl, window_right=wr, block_c=int(block_c),
                    kv_lens=kv, q=q, k=k, v=v, o=o, lse=l)
    _run(p, q, False, workspace)
    return o, l


def split_count(B: int, H: int, N: int, d: int, causal: bool = False, kv_lens: bool = False,
                num_splits: int = 0) -> int:
    """Number of key ranges the split-key forward uses for this call (1 = not split)."""
    p = attn_params(batch=B, heads=H, seqlen_q=N, head_dim=d, scale=1.0, causal=int(bool(causal)),
                    kv_lens=4096 if kv_lens else None, num_splits=int(num_splits))
    return int(load_library().fa_attn_fwd_splits(ctypes.byref(p)))


def split_workspace_size(B: int, H: int, N: int, d: int, causal: bool = False, kv_lens: bool = False,
                         num_splits: int = 0) -> int:
    p = attn_params(batch=B, heads=H, seqlen_q=N, head_dim=d, scale=1.0, causal=int(bool(causal)),
                    kv_lens=4096 if kv_lens else None, num_splits=int(num_splits))
    return int(load_library().fa_attn_fwd_workspace_size(ctypes.byref(p)))


def forward_split(q, k, v, causal: bool = False, scale: Optional[float] = None, kv_lens=None,
                  num_splits: int = 0, out: Optional[torch.Tensor] = None,
                  lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None
                  ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Split-key bf16 forward (FlashDecoding form): as forward(), with the key
    sequence of each query block cut into ranges merged by a second kernel.
    num_splits 0 = automatic, 1 = none, >= 2 = that many ranges per item."""
    _need_cuda(q, k, v)
    B, H, N, d = q.shape
    if q.dtype != torch.bfloat16 or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("forward_split takes bfloat16 q, k, v")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q.device)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    p = attn_params(batch=B, heads=H, seqlen_q=N, head_dim=d, scale=scale, causal=int(bool(causal)),
                    kv_lens=kv, num_splits=int(num_splits), q=q, k=k, v=v, o=o, lse=l)
    _run(p, q, False, workspace)
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


def _lists(row_ptr, col_idx, N):
    if row_ptr.dtype != torch.int32 or col_idx.dtype != torch.int32 or row_ptr.numel() != (N + 127) // 128 + 1:
        raise ValueError("row_ptr int32 [ceil(N/128) + 1], col_idx int32")


def forward_block_sparse(q, k, v, row_ptr, col_idx, causal: bool = False, scale: Optional[float] = None,
                         kv_lens=None, out: Optional[torch.Tensor] = None,
                         lse: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Block-sparse forward (128 x 128 blocks): query block i attends to the
    key blocks col_idx[row_ptr[i]:row_ptr[i+1]] only (see block_lists)."""
    _need_cuda(q, k, v, row_ptr, col_idx)
    if q.dtype != torch.bfloat16:
        raise ValueError("block lists take bfloat16 tensors")
    B, H, Hkv, N, d = _bhnd(q, k, v)
    _lists(row_ptr, col_idx, N)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q.device)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    p = attn_params(batch=B, heads=H, kv_heads=Hkv, seqlen_q=N, head_dim=d, scale=scale, causal=int(bool(causal)),
                    kv_lens=kv, block_row_ptr=row_ptr, block_col_idx=col_idx, q=q, k=k, v=v, o=o, lse=l)
    _run(p, q, False)
    return o, l


def backward_block_sparse(q, k, v, o, lse, dout, row_ptr, col_idx, causal: bool = False,
                          scale: Optional[float] = None, kv_lens=None, workspace: Optional[torch.Tensor] = None,
                          deterministic: bool = False):
    """Backward of forward_block_sparse: dQ [B,H,N,d], dK, dV [B,Hkv,N,d].
    deterministic: bitwise reproducible gradients (see backward)."""
    _need_cuda(q, k, v, o, lse, dout, row_ptr, col_idx)
    B, H, Hkv, N, d = _bhnd(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    p = attn_params(batch=B, heads=H, kv_heads=Hkv, seqlen_q=N, head_dim=d, scale=scale, causal=int(bool(causal)),
                    kv_lens=kv, block_row_ptr=row_ptr, block_col_idx=col_idx, deterministic=int(bool(deterministic)),
                    q=q, k=k, v=v, o=o, lse=lse, dout=dout, dq=dq, dk=dk, dv=dv)
    _run(p, q, True, workspace)
    return dq, dk, dv


def _rect(q, k, v):
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if (q.dtype != torch.bfloat16 or k.dtype != q.dtype or v.dtype != q.dtype or k.shape != (B, Hkv, Nk, d)
            or v.shape != k.shape or H % Hkv != 0):
        raise ValueError("q [B,H,Nq,d]; k, v [B,Hkv,Nk,d] bfloat16 with H a multiple of Hkv")
    return B, H, Hkv, Nq, Nk, d


def forward_rect(q, k, v, causal: bool = False, scale: Optional[float] = None, kv_lens=None,
                 num_splits: int = 0, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Nq queries against Nk keys (decoding against a key/value cache,
    cross-attention): q [B,H,Nq,d], k, v [B,Hkv,Nk,d] bf16.  Causal: the
    queries are the last Nq positions (query i sees keys j <= i + Nk - Nq)."""
    _need_cuda(q, k, v)
    B, H, Hkv, Nq, Nk, d = _rect(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q.device)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    p = attn_params(batch=B, heads=H, kv_heads=Hkv, seqlen_q=Nq, seqlen_k=Nk, head_dim=d, scale=scale,
                    causal=int(bool(causal)), kv_lens=kv, num_splits=int(num_splits), q=q, k=k, v=v, o=o, lse=l)
    _run(p, q, False, workspace)
    return o, l


def rect_split_count(B: int, H: int, Hkv: int, Nq: int, Nk: int, d: int, num_splits: int = 0) -> int:
    """Key ranges per item of the rectangular forward (1 = not split)."""
    p = attn_params(batch=B, heads=H, kv_heads=Hkv, seqlen_q=Nq, seqlen_k=Nk, head_dim=d, scale=1.0,
                    num_splits=int(num_splits))
    return int(load_library().fa_attn_fwd_splits(ctypes.byref(p)))


def backward_rect(q, k, v, o, lse, dout, causal: bool = False, scale: Optional[float] = None, kv_lens=None,
                  workspace: Optional[torch.Tensor] = None, deterministic: bool = False):
    """Backward of forward_rect: dQ [B,H,Nq,d], dK, dV [B,Hkv,Nk,d].
    deterministic: bitwise reproducible gradients (see backward)."""
    _need_cuda(q, k, v, o, lse, dout)
    B, H, Hkv, Nq, Nk, d = _rect(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    p = attn_params(batch=B, heads=H, kv_heads=Hkv, seqlen_q=Nq, seqlen_k=Nk, head_dim=d, scale=scale,
                    causal=int(bool(causal)), kv_lens=kv, deterministic=int(bool(deterministic)),
                    q=q, k=k, v=v, o=o, lse=lse, dout=dout, dq=dq, dk=dk, dv=dv)
    _run(p, q, True, workspace)
    return dq, dk, dv


def _cu(cu_seqlens, device):
    cu = cu_seqlens.to(device=device, dtype=torch.int32).contiguous()
    if cu.dim() != 1 or cu.numel() < 2:
        raise ValueError("cu_seqlens must be a 1-D tensor of batch + 1 offsets")
    return cu


def _packed(q, k, v, cu_seqlens_k):
    T, H, d = q.shape
    Hkv, Tk = k.shape[1], k.shape[0]
    if (q.dtype != torch.bfloat16 or k.dtype != q.dtype or v.dtype != q.dtype or k.shape != (Tk, Hkv, d)
            or v.shape != k.shape or H % Hkv != 0 or (cu_seqlens_k is None and Tk != T)):
        raise ValueError("q [total,H,d], k, v [total(_k),Hkv,d] bfloat16 with H a multiple of Hkv")
    return T, Tk, H, Hkv, d


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
    _need_cuda(q, k, v)
    T, Tk, H, Hkv, d = _packed(q, k, v, cu_seqlens_k)
    cu = _cu(cu_seqlens, q.device)
    cuk = None if cu_seqlens_k is None else _cu(cu_seqlens_k, q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((H, T), dtype=torch.float32, device=q.device) if lse is None else lse
    wl, wr = _window(window)
    p = attn_params(layout=FA_LAYOUT_PACKED, batch=cu.numel() - 1, heads=H, kv_heads=Hkv, seqlen_q=int(max_seqlen),
                    head_dim=d, total_q=T, total_k=Tk, scale=scale, causal=int(bool(causal)), window_left=wl,
                    window_right=wr, cu_seqlens_q=cu, cu_seqlens_k=cuk, q=q, k=k, v=v, o=o, lse=l)
    _run(p, q, False)
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
    _need_cuda(q, k, v)
    B, N, H, Hkv, d = _bnhd_shapes(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    p = attn_params(layout=FA_LAYOUT_BNHD, batch=B, heads=H, kv_heads=Hkv, seqlen_q=N, head_dim=d, scale=scale,
                    causal=int(bool(causal)), q=q, k=k, v=v, o=o, lse=l)
    _run(p, q, False)
    return o, l


def backward_bnhd(q, k, v, o, lse, dout, causal: bool = False, scale: Optional[float] = None,
                  workspace: Optional[torch.Tensor] = None, deterministic: bool = False):
    """dQ [B,N,H,d], dK, dV [B,N,Hkv,d] of forward_bnhd (dK, dV summed over
    the query heads sharing a key/value head).  deterministic: bitwise
    reproducible gradients (see backward)."""
    _need_cuda(q, k, v, o, lse, dout)
    B, N, H, Hkv, d = _bnhd_shapes(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    p = attn_params(layout=FA_LAYOUT_BNHD, batch=B, heads=H, kv_heads=Hkv, seqlen_q=N, head_dim=d, scale=scale,
                    causal=int(bool(causal)), deterministic=int(bool(deterministic)),
                    q=q, k=k, v=v, o=o, lse=lse, dout=dout, dq=dq, dk=dk, dv=dv)
    _run(p, q, True, workspace)
    return dq, dk, dv


def backward_varlen(q, k, v, o, lse, dout, cu_seqlens, max_seqlen: int, causal: bool = False,
                    scale: Optional[float] = None, workspace: Optional[torch.Tensor] = None,
                    deterministic: bool = False, cu_seqlens_k=None, max_seqlen_k: Optional[int] = None,
                    window: Optional[Tuple[int, int]] = None):
    """Backward of forward_varlen: dQ [total, H, d], dK, dV [total(_k), Hkv, d].
    deterministic: bitwise reproducible gradients (see backward).
    cu_seqlens_k / max_seqlen_k: separate key ranges (see forward_varlen)."""
    _need_cuda(q, k, v, o, lse, dout)
    T, Tk, H, Hkv, d = _packed(q, k, v, cu_seqlens_k)
    cu = _cu(cu_seqlens, q.device)
    cuk = None if cu_seqlens_k is None else _cu(cu_seqlens_k, q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    wl, wr = _window(window)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    mk = 0 if cu_seqlens_k is None else int(max_seqlen if max_seqlen_k is None else max_seqlen_k)
    p = attn_params(layout=FA_LAYOUT_PACKED, batch=cu.numel() - 1, heads=H, kv_heads=Hkv, seqlen_q=int(max_seqlen),
                    seqlen_k=mk, head_dim=d, total_q=T, total_k=Tk, scale=scale, causal=int(bool(causal)),
                    window_left=wl, window_right=wr, deterministic=int(bool(deterministic)), cu_seqlens_q=cu,
                    cu_seqlens_k=cuk, q=q, k=k, v=v, o=o, lse=lse, dout=dout, dq=dq, dk=dk, dv=dv)
    _run(p, q, True, workspace)
    return dq, dk, dv


def backward(q, k, v, o, lse, dout, causal: bool = False, scale: Optional[float] = None,
             kv_lens=None, workspace: Optional[torch.Tensor] = None,
             dq: Optional[torch.Tensor] = None, dk: Optional[torch.Tensor] = None,
             dv: Optional[torch.Tensor] = None, window: Optional[Tuple[int, int]] = None,
             deterministic: bool = False):
    """dQ, dK, dV of L = sum(O * dout).  With fewer key/value heads (k, v
    [B,Hkv,N,d]), dK and dV sum over the query heads sharing each one.
    window: the forward's sliding window (see forward).
    deterministic: bitwise-reproducible gradients (bf16): the dQ parts are
    added in key-block order."""
    _need_cuda(q, k, v, o, lse, dout)
    B, H, Hkv, N, d = _bhnd(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q.device)
    wl, wr = _window(window)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _need_cuda(dq, dk, dv)
    p = attn_params(dtype=_dtype(q), batch=B, heads=H, kv_heads=Hkv, seqlen_q=N, head_dim=d, scale=scale,
                    causal=int(bool(causal)), window_left=wl, window_right=wr,
                    deterministic=int(bool(deterministic)), kv_lens=kv,
                    q=q, k=k, v=v, o=o, lse=lse, dout=dout, dq=dq, dk=dk, dv=dv)
    _run(p, q, True, workspace)
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
    return forward_fp8_split(q8, k8, v8, sq, sk, sv, causal=causal, scale=scale, kv_lens=kv_lens,
                             num_splits=1, out=out, lse=lse)


def forward_fp8_split(q8, k8, v8, sq, sk, sv, causal: bool = False, scale: Optional[float] = None,
                      kv_lens=None, num_splits: int = 0, out: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None):
    """Split-key FP8 forward: forward_fp8 with the key ranges of forward_split."""
    _need_cuda(q8, k8, v8, sq, sk, sv)
    B, H, N, d = q8.shape
    Hkv = k8.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q8.device)
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q8.device) if lse is None else lse
    p = attn_params(dtype=FA_E4M3, batch=B, heads=H, kv_heads=Hkv, seqlen_q=N, head_dim=d, scale=scale,
                    causal=int(bool(causal)), kv_lens=kv, num_splits=int(num_splits), q=q8, k=k8, v=v8,
                    q_scale=sq, k_scale=sk, v_scale=sv, o=o, lse=l)
    _run(p, q8, False, workspace)
    return o, l


def backward_fp8(q8, k8, v8, sq, sk, sv, o, lse, dout, causal: bool = False, scale: Optional[float] = None,
                 kv_lens=None, workspace: Optional[torch.Tensor] = None):
    """FP8 backward (d = 128) of forward_fp8: q8, k8, v8 E4M3 codes [B,H,N,128]
    with their block scales, the forward's o (bf16) and lse, and the bf16
    upstream gradient dout.  The five products run on FP8 tensor cores (dS in
    E5M2); returns float32 dQ, dK, dV [B,H,N,128]."""
    _need_cuda(q8, k8, v8, sq, sk, sv, o, lse, dout)
    B, H, N, d = q8.shape
    if k8.shape != q8.shape or v8.shape != q8.shape or dout.dtype != torch.bfloat16:
        raise ValueError("q8, k8, v8 [B,H,N,128] E4M3 codes; dout bfloat16")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kv = _kv(kv_lens, B, q8.device)
    dq, dk, dv = (torch.empty((B, H, N, d), dtype=torch.float32, device=q8.device) for _ in range(3))
    p = attn_params(dtype=FA_E4M3, batch=B, heads=H, seqlen_q=N, head_dim=d, scale=scale, causal=int(bool(causal)),
                    kv_lens=kv, q=q8, k=k8, v=v8, q_scale=sq, k_scale=sk, v_scale=sv, o=o, lse=lse, dout=dout,
                    dq=dq, dk=dk, dv=dv)
    _run(p, q8, True, workspace)
    return dq, dk, dv


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
