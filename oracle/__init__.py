"""CPU oracle for exact tiled attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
product path never imports it, and the two share no code: the arithmetic lives
in ``oracle.c`` (plain fp64 C, naive loops), compiled with gcc into
``liboracle.so`` next to this file.

Entry points and what pins each one (tests/test_oracle_*.py):

* ``fwd`` / ``bwd`` -- materialised attention and its gradients, one head at a
  time.  Pinned by: the six-score closed forms evaluated in 50-digit mpmath
  (attention-kernels wiki, §02 block ledger), the 5-position causal example's
  closed forms (same page, §04), float64 autograd of the materialised formula
  (an independent derivation of the gradients), central finite differences,
  the single-visible-key and constant-score closed forms, sum_j P_ij = 1,
  D = rowsum(dO*O), key-shift invariance (sum_j dS_ij = 0) and the
  fully-masked-row convention.
* ``fwd_rows`` / ``bwd_rows`` -- the same definitions row by row, for shapes
  whose N x N matrices do not fit.  Pinned against ``fwd`` / ``bwd``.
* the sliding window (``window=(left, right)`` on the four functions above,
  chapter 18 §18.7.1 window_size).  Pinned by: float64 autograd of the
  materialised formula with an explicit additive mask, the window (0, 0)
  closed form (each query sees only its own key: O_i = v_i, LSE_i = S_ii,
  dQ = dK = 0, dV_i = dO_i), window (-1, 0) equal to the causal mask,
  windows wider than N equal to no window, and central finite differences.
* ``fwd_rect`` / ``bwd_rect`` -- rectangular attention (Nq queries, Nk keys: decoding
  against a key/value cache, cross-attention; chapter 18 §18.8.2), causal
  with the queries as the last Nq positions.  Pinned by: Nq = Nk equal to
  ``fwd`` exactly, the causal case equal to the last Nq rows of ``fwd`` on
  the full Nk-row sequence exactly, float64 torch softmax with an explicit
  mask, and the one-query closed form (LSE = logsumexp of its scores);
  the backward by float64 autograd with the same mask, Nq = Nk equal to
  ``bwd`` exactly, and central finite differences.
* the block-sparse mask (``block_mask`` [nb][nb] of 0/1 over block_size
  blocks, chapter 18 §18.8.1).  Pinned by: float64 autograd with the mask
  expanded to elements by a Kronecker product, the all-ones mask equal to no
  mask, the block-diagonal mask equal to independent attention on each block
  (separate oracle calls on the slices), a row of blocks with no entry giving
  O = 0 / LSE = -inf / zero gradients, and central finite differences.
* ``tiled_fwd`` / ``tiled_bwd`` -- Algorithms 1 and 2 of the FA-v2 analysis
  page (§4, §5.4) with arbitrary Br/Bc.  Pinned against ``fwd`` / ``bwd`` on
  the pages' worked shapes (N=4,d=3,Br=Bc=2; the 5-position example with 2x2
  blocks; every block size of the six-score row).
* ``quantize_fp8`` / ``e4m3_encode`` / ``e4m3_decode`` -- per-block E4M3
  quantisation (chapter 18 §18.6.2).  Pinned against torch's float8_e4m3fn
  conversion on every in-range fp32 bucket, the format's closed-form codes,
  and saturation.

No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)
_ip = ctypes.POINTER(ctypes.c_int)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (fp64, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-D_GNU_SOURCE",
               "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            _i = ctypes.c_int
            lib.oracle_fwd_mask.argtypes = [_dp, _dp, _dp, _dp, _dp, _i, _i, _i, _i, ctypes.c_double,
                                            _i, _i, _i, _u8p, _i, _ip, _i]
            lib.oracle_bwd_mask.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp,
                                            _i, _i, _i, _i, ctypes.c_double, _i, _i, _i, _u8p, _i, _ip, _i]
            lib.oracle_fwd_rows_mask.argtypes = [_dp, _dp, _dp, _i, _i, ctypes.c_double, _i, _i, _i, _i,
                                                 _u8p, _i, _ip, _i, _dp, _dp]
            lib.oracle_bwd_rows_mask.argtypes = [_dp, _dp, _dp, _dp, _i, _i, ctypes.c_double, _i, _i, _i,
                                                 _i, _u8p, _i, _ip, _i, _dp, _ip, _i, _dp, _dp, _dp, _dp, _i]
            lib.oracle_tiled_fwd.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                             ctypes.c_int, _ip, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int]
            lib.oracle_tiled_bwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_double, ctypes.c_int, _ip,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int]
            lib.oracle_fwd_rect.argtypes = [_dp, _dp, _dp, _dp, _dp, _i, _i, _i, _i, _i, ctypes.c_double, _i,
                                            _ip, _i]
            lib.oracle_bwd_rect.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _i, _i, _i, _i, _i,
                                            ctypes.c_double, _i, _ip, _i]
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_quantize_fp8.argtypes = [_fp, _u8p, _fp, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int]
            lib.oracle_default_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor -> exact float64 copy
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a: np.ndarray, ct):
    return a.ctypes.data_as(ct)


def _kv(kv_lens, B):
    if kv_lens is None:
        return None, None
    arr = np.ascontiguousarray(np.asarray(
        kv_lens.cpu().numpy() if hasattr(kv_lens, "cpu") else kv_lens, dtype=np.int32))
    assert arr.shape == (B,)
    return arr, _ptr(arr, _ip)


def _win(window):
    """(left, right) of the sliding window; -1 (or None) = no bound on that side."""
    if window is None:
        return -1, -1
    wl, wr = window
    return (-1 if wl is None or wl < 0 else int(wl)), (-1 if wr is None or wr < 0 else int(wr))


def _bm(block_mask, block_size, N):
    """(array, pointer, block size) of a 0/1 block mask [ceil(N/bs)][ceil(N/bs)]."""
    if block_mask is None:
        return None, None, 0
    bs = int(block_size)
    nb = (N + bs - 1) // bs
    arr = np.ascontiguousarray(np.asarray(block_mask, dtype=np.uint8) != 0, dtype=np.uint8)
    assert arr.shape == (nb, nb), (arr.shape, nb)
    return arr, _ptr(arr, _u8p), bs


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def fwd(q, k, v, scale, causal=False, kv_lens=None, nthreads=0, window=None, block_mask=None,
        block_size=128):
    """Materialised forward. q,k,v: [B,H,N,d]. Returns (O [B,H,N,d], LSE [B,H,N]) fp64.

    window = (left, right): key j is visible to query i only if
    i - left <= j <= i + right (chapter 18 §18.7.1 window_size; -1 = unbounded).
    block_mask: 0/1 [nb][nb] over block_size x block_size blocks; key j is
    visible to query i only if block_mask[i // bs][j // bs] (§18.8.1)."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    o = np.zeros_like(q)
    lse = np.zeros((B, H, N))
    kv, kvp = _kv(kv_lens, B)
    bma, bmp, bs = _bm(block_mask, block_size, N)
    rc = lib.oracle_fwd_mask(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(o, _dp), _ptr(lse, _dp),
                             B, H, N, d, float(scale), int(bool(causal)), *_win(window), bmp, bs, kvp,
                             int(nthreads))
    assert rc == 0
    return o, lse


def bwd(q, k, v, dout, scale, causal=False, kv_lens=None, nthreads=0, window=None, block_mask=None,
        block_size=128):
    """Materialised backward of L = sum(O*dO).

    Returns dict with o, lse, dq, dk, dv, D (D by its definition sum_j P dP)."""
    lib = _load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, N, d = q.shape
    o, dq, dk, dv = (np.zeros_like(q) for _ in range(4))
    lse = np.zeros((B, H, N))
    D = np.zeros((B, H, N))
    kv, kvp = _kv(kv_lens, B)
    bma, bmp, bs = _bm(block_mask, block_size, N)
    rc = lib.oracle_bwd_mask(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(dout, _dp), _ptr(o, _dp),
                             _ptr(lse, _dp), _ptr(dq, _dp), _ptr(dk, _dp), _ptr(dv, _dp),
                             _ptr(D, _dp), B, H, N, d, float(scale), int(bool(causal)), *_win(window),
                             bmp, bs, kvp, int(nthreads))
    assert rc == 0
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv, D=D)


def fwd_rect(q, k, v, scale, causal=False, kv_lens=None, nthreads=0):
    """Rectangular forward: q [B,H,Nq,d], k, v [B,H,Nk,d].  Causal: the queries
    are the last Nq positions, query i sees keys j <= i + Nk - Nq.
    Returns (O [B,H,Nq,d], LSE [B,H,Nq]) fp64."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    assert k.shape == (B, H, Nk, d) and v.shape == k.shape
    o = np.zeros_like(q)
    lse = np.zeros((B, H, Nq))
    kv, kvp = _kv(kv_lens, B)
    rc = lib.oracle_fwd_rect(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(o, _dp), _ptr(lse, _dp), B, H, Nq,
                             Nk, d, float(scale), int(bool(causal)), kvp, int(nthreads))
    assert rc == 0
    return o, lse


def bwd_rect(q, k, v, dout, scale, causal=False, kv_lens=None, nthreads=0):
    """Backward of fwd_rect (L = sum(O * dout)): dict dq [B,H,Nq,d], dk, dv [B,H,Nk,d]."""
    lib = _load()
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    assert k.shape == (B, H, Nk, d) and v.shape == k.shape and g.shape == q.shape
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    kv, kvp = _kv(kv_lens, B)
    rc = lib.oracle_bwd_rect(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(g, _dp), _ptr(dq, _dp),
                             _ptr(dk, _dp), _ptr(dv, _dp), B, H, Nq, Nk, d, float(scale), int(bool(causal)),
                             kvp, int(nthreads))
    assert rc == 0
    return dict(dq=dq, dk=dk, dv=dv)


def fwd_rows(q_head, k_head, v_head, scale, causal, kv_len, rows, window=None, block_mask=None,
             block_size=128):
    """Row-sampled forward of ONE head ([N,d] inputs). Returns (O_rows, LSE_rows)."""
    lib = _load()
    q, k, v = _f64(q_head), _f64(k_head), _f64(v_head)
    N, d = q.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    o = np.zeros((len(rows), d))
    lse = np.zeros(len(rows))
    bma, bmp, bs = _bm(block_mask, block_size, N)
    rc = lib.oracle_fwd_rows_mask(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), N, d, float(scale),
                                  int(bool(causal)), int(kv_len), *_win(window), bmp, bs, _ptr(rows, _ip),
                                  len(rows), _ptr(o, _dp), _ptr(lse, _dp))
    assert rc == 0
    return o, lse


def bwd_rows(q_head, k_head, v_head, dout_head, scale, causal, kv_len, rows, keys, nthreads=0,
             window=None, block_mask=None, block_size=128):
    """Row-sampled backward of ONE head. Returns dict dq (rows), dk, dv (keys), lse, D (all rows)."""
    lib = _load()
    q, k, v, g = _f64(q_head), _f64(k_head), _f64(v_head), _f64(dout_head)
    N, d = q.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    keys = np.ascontiguousarray(np.asarray(keys, dtype=np.int32))
    dq = np.zeros((len(rows), d))
    dk = np.zeros((max(len(keys), 1), d))
    dv = np.zeros((max(len(keys), 1), d))
    lse = np.zeros(N)
    D = np.zeros(N)
    bma, bmp, bs = _bm(block_mask, block_size, N)
    rc = lib.oracle_bwd_rows_mask(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(g, _dp), N, d,
                                  float(scale), int(bool(causal)), int(kv_len), *_win(window), bmp, bs,
                                  _ptr(rows, _ip), len(rows), _ptr(dq, _dp), _ptr(keys, _ip), len(keys),
                                  _ptr(dk, _dp), _ptr(dv, _dp), _ptr(lse, _dp), _ptr(D, _dp),
                                  int(nthreads))
    assert rc == 0
    return dict(dq=dq, dk=dk[:len(keys)], dv=dv[:len(keys)], lse=lse, D=D)


def tiled_fwd(q, k, v, scale, causal=False, kv_lens=None, Br=2, Bc=2, nthreads=0):
    """Algorithm 1 (FA-v2 analysis page, §4), fp64. Returns (O, LSE)."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    o = np.zeros_like(q)
    lse = np.zeros((B, H, N))
    kv, kvp = _kv(kv_lens, B)
    rc = lib.oracle_tiled_fwd(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(o, _dp),
                              _ptr(lse, _dp), B, H, N, d, float(scale), int(bool(causal)), kvp,
                              int(Br), int(Bc), int(nthreads))
    assert rc == 0
    return o, lse


def tiled_bwd(q, k, v, o, lse, dout, scale, causal=False, kv_lens=None, Br=2, Bc=2, nthreads=0):
    """Algorithm 2 (FA-v2 analysis page, §5.4), fp64. Returns (dQ, dK, dV)."""
    lib = _load()
    q, k, v, o, lse, g = _f64(q), _f64(k), _f64(v), _f64(o), _f64(lse), _f64(dout)
    B, H, N, d = q.shape
    dq, dk, dv = (np.zeros_like(q) for _ in range(3))
    kv, kvp = _kv(kv_lens, B)
    rc = lib.oracle_tiled_bwd(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(o, _dp),
                              _ptr(lse, _dp), _ptr(g, _dp), _ptr(dq, _dp), _ptr(dk, _dp),
                              _ptr(dv, _dp), B, H, N, d, float(scale), int(bool(causal)), kvp,
                              int(Br), int(Bc), int(nthreads))
    assert rc == 0
    return dq, dk, dv


def e4m3_encode(x: float) -> int:
    return int(_load().oracle_e4m3_encode(ctypes.c_float(x)))


def e4m3_decode(code: int) -> float:
    return float(_load().oracle_e4m3_decode(ctypes.c_uint8(code)))


def e4m3_decode_array(codes: np.ndarray) -> np.ndarray:
    table = np.array([e4m3_decode(c) for c in range(256)])
    return table[np.asarray(codes, dtype=np.uint8)]


def quantize_fp8(x, blk=64):
    """Per-(b,h, blk rows x d) E4M3 quantisation. x: [B,H,N,d] bf16-representable.

    Returns (codes uint8 [B,H,N,d], scales float32 [B,H,ceil(N/blk)])."""
    lib = _load()
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").float().numpy()
    x = np.ascontiguousarray(x, dtype=np.float32)
    B, H, N, d = x.shape
    nb = (N + blk - 1) // blk
    codes = np.zeros(x.shape, dtype=np.uint8)
    scales = np.zeros((B, H, nb), dtype=np.float32)
    rc = lib.oracle_quantize_fp8(_ptr(x, _fp), _ptr(codes, _u8p), _ptr(scales, _fp), B, H, N, d,
                                 int(blk))
    assert rc == 0
    return codes, scales


def dequantize_fp8(codes, scales, blk=64):
    """Exact fp64 value of each quantised element: s_block * decode(code)."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.float64)
    B, H, N, d = codes.shape
    vals = e4m3_decode_array(codes)
    rowblk = np.arange(N) // blk
    return vals * scales[:, :, rowblk][..., None]
