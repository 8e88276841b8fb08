"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no attention arithmetic: it only draws numbers.  Every
tensor is drawn as fp32 N(0, 1) from a CPU ``torch.Generator`` seeded per
tensor (q=1, k=2, v=3 by default), multiplied by an optional magnitude (the
large-value stress case uses 8 for q and k and 100 for v), and rounded to
bf16 with round-to-nearest-even.  Both sides then read the same bf16 bits.

Shapes follow the geometry of the chowfi/kernels README ("Result" section:
batch 1, 32 query heads, 8 KV heads, head size 128) in sequence-major BSHD
layout: q/out [1,S,32,128], k/v [1,S,8,128]; decode q/out [1,1,32,128],
kcache/vcache [1,L,8,128].
"""
from __future__ import annotations

import torch

HQ = 32
HKV = 8
HEAD_DIM = 128

SEED_Q, SEED_K, SEED_V = 1, 2, 3
STRESS_QK, STRESS_V = 8.0, 100.0


def normal_bf16(shape, seed: int, magnitude: float = 1.0) -> torch.Tensor:
    """fp32 N(0,1) from ``seed`` times ``magnitude``, rounded to bf16 (RNE)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if magnitude != 1.0:
        x.mul_(magnitude)
    return x.to(torch.bfloat16)


def prefill_inputs(S: int, stress: bool = False, hq: int = HQ, hkv: int = HKV,
                   d: int = HEAD_DIM, seeds=(SEED_Q, SEED_K, SEED_V)):
    """(q, k, v) CPU bf16 tensors for a prefill of length S, batch 1."""
    mq = STRESS_QK if stress else 1.0
    mv = STRESS_V if stress else 1.0
    q = normal_bf16((1, S, hq, d), seeds[0], mq)
    k = normal_bf16((1, S, hkv, d), seeds[1], mq)
    v = normal_bf16((1, S, hkv, d), seeds[2], mv)
    return q, k, v


def decode_inputs(L: int, stress: bool = False, hq: int = HQ, hkv: int = HKV,
                  d: int = HEAD_DIM, seeds=(SEED_Q, SEED_K, SEED_V)):
    """(q, kcache, vcache) CPU bf16 tensors for one decode token, batch 1."""
    mq = STRESS_QK if stress else 1.0
    mv = STRESS_V if stress else 1.0
    q = normal_bf16((1, 1, hq, d), seeds[0], mq)
    kc = normal_bf16((1, L, hkv, d), seeds[1], mq)
    vc = normal_bf16((1, L, hkv, d), seeds[2], mv)
    return q, kc, vc
