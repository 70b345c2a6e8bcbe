"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws random tensors and
names the workload shapes.  Both the CUDA path and the CPU oracle consume the
SAME bf16-rounded tensors it returns (the oracle upcasts them exactly to fp64).

Workloads (chapter 18 of the FlashAttention book uses B, H, N, d shapes of this
kind for its timing tables; every value here is drawn from N(0, 1)):

  tiny      B=1 H=1  N=128   d=64   seed 1001  (fp32 and bf16; causal 0/1)
  mid       B=4 H=16 N=2048  d=64   seed 1002  (causal 0/1)
  long_head B=2 H=16 N=4096  d=128  seed 1003  (causal fwd+bwd, non-causal fwd)
  ragged    B=8 H=32 N=1024  d=128  seed 1004  kv_len ~ U{1..1024}, kv_len[0] = 0
  long_seq  B=1 H=8  N=16384 d=128  seed 1005  (bf16 causal; FP8 non-causal)
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    seed: int
    ragged: bool = False

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 128, 64, 1001),
    "mid": Workload("mid", 4, 16, 2048, 64, 1002),
    "long_head": Workload("long_head", 2, 16, 4096, 128, 1003),
    "ragged": Workload("ragged", 8, 32, 1024, 128, 1004, ragged=True),
    "long_seq": Workload("long_seq", 1, 8, 16384, 128, 1005),
}


def randn_on_device(shape, seed: int, device, dtype=torch.bfloat16) -> torch.Tensor:
    """N(0,1) drawn by the device's own generator (seeded), for tensors too
    large to draw on the host; the oracle then reads the sampled parts of the
    same tensor."""
    g = torch.Generator(device=device).manual_seed(int(seed))
    return torch.randn(*shape, generator=g, dtype=torch.float32, device=device).to(dtype)


def randn(shape, seed: int, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """N(0,1) drawn in fp32 on the CPU generator, then cast (so every device
    and dtype sees the same underlying draw)."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    return x.to(dtype).to(device)


def qkv(B, H, N, d, seed, dtype=torch.bfloat16, device="cpu", with_dout=True):
    """Q, K, V (and dO) of shape [B,H,N,d]; streams seed, seed+1, ... ."""
    shape = (B, H, N, d)
    q = randn(shape, seed, dtype, device)
    k = randn(shape, seed + 1, dtype, device)
    v = randn(shape, seed + 2, dtype, device)
    if not with_dout:
        return q, k, v
    do = randn(shape, seed + 3, dtype, device)
    return q, k, v, do


def kv_lens_ragged(B: int, N: int, seed: int, device="cpu") -> torch.Tensor:
    """Per-sequence valid key length ~ U{1..N}; item 0 forced to 0 (all rows masked)."""
    g = torch.Generator(device="cpu").manual_seed(int(seed) + 100)
    kv = torch.randint(1, N + 1, (B,), generator=g, dtype=torch.int32)
    kv[0] = 0
    return kv.to(device)


def workload_inputs(w: Workload, dtype=torch.bfloat16, device="cpu", with_dout=True):
    t = qkv(w.B, w.H, w.N, w.d, w.seed, dtype, device, with_dout)
    kv: Optional[torch.Tensor] = kv_lens_ragged(w.B, w.N, w.seed, device) if w.ragged else None
    return t, kv
