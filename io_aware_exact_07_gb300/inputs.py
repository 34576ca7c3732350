"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and builds the workload descriptions;
it holds none of the attention arithmetic. Both the GPU path and the CPU
oracle consume what it produces.

Recipe (one CPU ``torch.Generator`` seeded with ``seed``):
  Q, K, V, dO drawn in that order as ``randn(B, H, N, d)`` in fp32 (K and V
  with H_kv heads for grouped-query attention), then rounded to bf16; for the
  key-padding workload the per-sequence valid key
  lengths are drawn next as ``randint(lo, hi + 1, (B,))``. The dropout Philox
  stream uses (seed, offset) = (0, 0). The block-sparse workload's mask is the
  deterministic butterfly pattern built by the library itself.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool = False
    dropout_p: float = 0.0
    padding: tuple | None = None  # (lo, hi) inclusive range of valid key lengths
    butterfly: bool = False
    seed: int = 0
    Hkv: int | None = None  # K/V heads (grouped-query attention); None: one per query head
    window: tuple = (-1, -1)  # sliding window (left, right); -1: that side unbounded
    description: str = field(default="", compare=False)

    @property
    def kv_heads(self) -> int:
        return self.H if self.Hkv is None else self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# The five workloads of the benchmark suite (shapes of the pages' experiments:
# GPT-2-medium attention, long-context LRA / Path-X lengths, block-sparse).
TINY = Workload("tiny", 1, 1, 128, 64,
                description="B=1 H=1 N=128 d=64, non-causal, no dropout")
GPT2_MEDIUM = Workload("gpt2_medium", 64, 16, 1024, 64, dropout_p=0.1, padding=(512, 1024),
                       description="B=64 H=16 N=1024 d=64, key padding U[512,1024], dropout 0.1")
CAUSAL = Workload("causal_4k", 8, 32, 4096, 128, causal=True,
                  description="B=8 H=32 N=4096 d=128, causal")
LONG_D64 = Workload("long_16k_d64", 1, 16, 16384, 64,
                    description="B=1 H=16 N=16384 d=64, non-causal")
LONG_D128 = Workload("long_16k_d128", 1, 16, 16384, 128,
                     description="B=1 H=16 N=16384 d=128, non-causal")
SPARSE = Workload("butterfly_16k", 4, 16, 16384, 64, butterfly=True,
                  description="B=4 H=16 N=16384 d=64, butterfly block mask, 128x128 blocks")

# Grouped-query attention (K/V heads shared by query heads, which the page on
# FlashAttention and its successors names as a further cut of K/V reads),
# measured beyond the five workloads: the causal decoder shape with 4 query
# heads per K/V head.
GQA_CAUSAL = Workload("gqa_causal_4k", 8, 32, 4096, 128, causal=True, Hkv=8,
                      description="B=8 H=32 H_kv=8 N=4096 d=128, causal, grouped K/V heads")

# Sliding-window (local) attention, which the pages list among the variants
# and the block-skipping patterns without a workload: a long causal sequence
# where each query sees the 4096 keys ending at itself.
SLIDING = Workload("sliding_16k", 2, 32, 16384, 128, causal=True, window=(4095, -1),
                   description="B=2 H=32 N=16384 d=128, causal, sliding window of 4096 keys")

ALL = {w.name: w for w in (TINY, GPT2_MEDIUM, CAUSAL, LONG_D64, LONG_D128, SPARSE, GQA_CAUSAL,
                           SLIDING)}


def draw(w: Workload, with_grad: bool = True):
    """Return dict with bf16 CPU tensors q, k, v, (do) and int32 seqlens (or None)."""
    g = torch.Generator().manual_seed(w.seed)
    out = {}
    names = ("q", "k", "v", "do") if with_grad else ("q", "k", "v")
    for name in names:
        heads = w.kv_heads if name in ("k", "v") else w.H
        out[name] = torch.randn((w.B, heads, w.N, w.d), generator=g,
                                dtype=torch.float32).to(torch.bfloat16)
    if w.padding is not None:
        lo, hi = w.padding
        out["seqlens"] = torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int64).to(
            torch.int32)
    else:
        out["seqlens"] = None
    return out


@dataclass(frozen=True)
class DecodeWorkload:
    """Nq new query rows per head over a K/V cache of Nk rows (forward only)."""
    name: str
    B: int
    H: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    causal: bool = False
    lengths: tuple | None = None  # (lo, hi) inclusive range of valid cache lengths
    seed: int = 0
    description: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# Decode: the pages name single-token decode as memory-bound and left
# unoptimised by the FlashAttention kernels, without a workload; this one is a
# serving-shaped step of one new token per sequence over a 16K-token cache,
# grouped K/V heads (4 query heads each), K/V 1.07 GB (well above L2).
DECODE = DecodeWorkload("decode_16k", 16, 32, 8, 1, 16384, 128,
                        description="B=16 H=32 H_kv=8 Nq=1 Nk=16384 d=128, one new token per "
                                    "sequence over a full 16K K/V cache")


def draw_decode(w: DecodeWorkload) -> dict:
    """bf16 CPU tensors q [B,H,Nq,d], k, v [B,Hkv,Nk,d] drawn in that order as
    randn in fp32, then int32 cache lengths if w.lengths is set, else None."""
    g = torch.Generator().manual_seed(w.seed)
    out = {"q": torch.randn((w.B, w.H, w.Nq, w.d), generator=g).to(torch.bfloat16)}
    for name in ("k", "v"):
        out[name] = torch.randn((w.B, w.Hkv, w.Nk, w.d), generator=g).to(torch.bfloat16)
    if w.lengths is not None:
        lo, hi = w.lengths
        out["seqlens"] = torch.randint(lo, hi + 1, (w.B,), generator=g,
                                       dtype=torch.int64).to(torch.int32)
    else:
        out["seqlens"] = None
    return out


def draw_small(B, H, N, d, seed=0, with_grad=True, padding=None):
    """Same recipe for an ad-hoc shape (parity cases and edge cases)."""
    w = Workload("adhoc", B, H, N, d, padding=padding, seed=seed)
    return draw(w, with_grad=with_grad)


def sample_heads(w: Workload, count: int = 4, seed: int = 1234):
    """Deterministic subset of (b, h) heads: first, last and seeded others."""
    heads = [(0, 0), (w.B - 1, w.H - 1)]
    g = torch.Generator().manual_seed(seed)
    while len(heads) < min(count, w.B * w.H):
        idx = int(torch.randint(0, w.B * w.H, (1,), generator=g))
        hb = (idx // w.H, idx % w.H)
        if hb not in heads:
            heads.append(hb)
    return heads


# FP8 forward: the causal decoder shape, bf16 inputs quantised by the library.
FP8_CAUSAL = Workload("fp8_causal_4k", 8, 32, 4096, 128, causal=True,
                      description="B=8 H=32 N=4096 d=128, causal, FP8 (e4m3) forward with "
                                  "Hadamard rotation")


def rotation_signs(d: int, seed: int = 0) -> torch.Tensor:
    """+-1 fp32 [d]: the random signs of the FP8 path's rotation, drawn once."""
    g = torch.Generator().manual_seed(seed)
    return (torch.randint(0, 2, (d,), generator=g) * 2 - 1).to(torch.float32)


def draw_fp8_codes(B, H, N, d, seed=0):
    """Random e4m3 codes for the FP8 forward: q8, k8, v8 uint8 [B, H, N, d] as the
    bytes of N(0, 1) * 64 rounded to e4m3 by torch (magnitudes up to ~300, so
    most of the code range is used), and positive scales s_q, s_k [B, H],
    s_v [B, H, d] drawn uniformly from [0.003, 0.012]."""
    g = torch.Generator().manual_seed(seed)
    out = {}
    for name in ("q8", "k8", "v8"):
        x = torch.randn((B, H, N, d), generator=g) * 64.0
        out[name] = x.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    out["s_q"] = torch.rand((B, H), generator=g) * 0.009 + 0.003
    out["s_k"] = torch.rand((B, H), generator=g) * 0.009 + 0.003
    out["s_v"] = torch.rand((B, H, d), generator=g) * 0.009 + 0.003
    return out
