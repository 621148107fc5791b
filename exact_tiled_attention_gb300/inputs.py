"""Seeded synthetic inputs for the attention workloads.

This module holds no attention arithmetic: it only draws i.i.d. N(0, 1)
tensors (and decode valid lengths) from a seeded torch generator, in the
order q, k, v (then lengths), and rounds them to the workload's dtype.  The
GPU tests and the oracle consume the SAME rounded tensors.

The shapes are those of the workloads the pages discuss: a tiny fp16 forward,
the [1, 8, 4096, 64] fp16 non-causal shape timed in "Learning FlashAttention
the Hard Way — Part 2", a causal bf16 [4, 16, 8192, 128] prefill, a GQA causal
prefill (32 query heads over 8 KV heads) and a 64-sequence one-query decode
over a 32768-slot KV cache split into 16 chunks.
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
    Hkv: int
    Sq: int
    Sk: int
    d: int
    dtype: torch.dtype
    causal: bool
    decode: bool = False
    n_split: int = 0
    len_lo: int = 0          # decode: valid lengths uniform on [len_lo, len_hi]
    len_hi: int = 0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


WORKLOADS = {
    "tiny_fwd_fp16": Workload("tiny_fwd_fp16", 1, 4, 4, 128, 128, 64, torch.float16, False, seed=1),
    "prefill_fp16_b1_h8_s4096_d64": Workload("prefill_fp16_b1_h8_s4096_d64", 1, 8, 8, 4096, 4096, 64,
                                             torch.float16, False, seed=2),
    "causal_bf16_b4_h16_s8192_d128": Workload("causal_bf16_b4_h16_s8192_d128", 4, 16, 16, 8192, 8192,
                                              128, torch.bfloat16, True, seed=3),
    "noncausal_bf16_b4_h16_s8192_d128": Workload("noncausal_bf16_b4_h16_s8192_d128", 4, 16, 16, 8192,
                                                 8192, 128, torch.bfloat16, False, seed=6),
    "gqa_causal_bf16_b2_hq32_hkv8_s4096_d128": Workload("gqa_causal_bf16_b2_hq32_hkv8_s4096_d128", 2,
                                                        32, 8, 4096, 4096, 128, torch.bfloat16, True,
                                                        seed=4),
    "decode_splitkv_bf16_b64_hq32_hkv8_sk32768_d128": Workload(
        "decode_splitkv_bf16_b64_hq32_hkv8_sk32768_d128", 64, 32, 8, 1, 32768, 128, torch.bfloat16,
        False, decode=True, n_split=16, len_lo=1024, len_hi=32768, seed=5),
}


def make_generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn(shape, dtype, gen, device):
    """i.i.d. N(0,1) drawn in fp32, then rounded to `dtype`."""
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


def make_prefill(B, H, Hkv, Sq, Sk, d, dtype, seed, device="cpu"):
    """q [B,H,Sq,d], k/v [B,Hkv,Sk,d], drawn in that order."""
    g = make_generator(seed, device)
    q = randn((B, H, Sq, d), dtype, g, device)
    k = randn((B, Hkv, Sk, d), dtype, g, device)
    v = randn((B, Hkv, Sk, d), dtype, g, device)
    return q, k, v


def make_decode(B, Hq, Hkv, Sk_max, d, dtype, len_lo, len_hi, seed, device="cpu"):
    """q [B,Hq,1,d], k/v caches [B,Hkv,Sk_max,d], then int32 valid lengths
    uniform on [len_lo, len_hi] inclusive."""
    g = make_generator(seed, device)
    q = randn((B, Hq, 1, d), dtype, g, device)
    k = randn((B, Hkv, Sk_max, d), dtype, g, device)
    v = randn((B, Hkv, Sk_max, d), dtype, g, device)
    seqlens = torch.randint(len_lo, len_hi + 1, (B,), generator=g, device=device,
                            dtype=torch.int64).to(torch.int32)
    return q, k, v, seqlens


def make_workload(w: Workload, device="cpu"):
    if w.decode:
        return make_decode(w.B, w.H, w.Hkv, w.Sk, w.d, w.dtype, w.len_lo, w.len_hi, w.seed, device)
    return make_prefill(w.B, w.H, w.Hkv, w.Sq, w.Sk, w.d, w.dtype, w.seed, device)
