"""Seeded synthetic inputs for retention workloads.

This module only draws random numbers; it holds none of the method's
arithmetic (no decay, no scaling, no products).  Both the CUDA parity tests
and the CPU oracle read their inputs from here, so the two sides see the same
values.  Every tensor is drawn on the CPU with a seeded ``torch.Generator`` in
fp32 and then rounded to the requested dtype (round-to-nearest-even for
bf16), so a given (shape, seed, dtype) always yields the same bits.
"""
from __future__ import annotations

import torch


def normal(shape, seed: int, dtype=torch.float32, std: float = 1.0) -> torch.Tensor:
    """iid N(0, std^2) CPU tensor of `shape`, drawn in fp32 then cast."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(dtype)


def qkv(B: int, H: int, N: int, dk: int, dv: int, seed: int, dtype=torch.bfloat16):
    """Q, K: [B,H,N,dk]; V: [B,H,N,dv]; iid N(0,1), three independent streams."""
    q = normal((B, H, N, dk), 3 * seed + 0, dtype)
    k = normal((B, H, N, dk), 3 * seed + 1, dtype)
    v = normal((B, H, N, dv), 3 * seed + 2, dtype)
    return q, k, v


def decode_steps(T: int, B: int, H: int, dk: int, dv: int, seed: int, dtype=torch.bfloat16):
    """Per-step q, k: [T,B,H,dk]; v: [T,B,H,dv]; iid N(0,1)."""
    q = normal((T, B, H, dk), 7919 + 3 * seed + 0, dtype)
    k = normal((T, B, H, dk), 7919 + 3 * seed + 1, dtype)
    v = normal((T, B, H, dv), 7919 + 3 * seed + 2, dtype)
    return q, k, v


def decode_state(B: int, H: int, dk: int, dv: int, seed: int, std: float = 0.1) -> torch.Tensor:
    """Initial fp32 state [B,H,dk,dv] ~ N(0, std^2) (std 0.1 for the decode workload)."""
    return normal((B, H, dk, dv), 104729 + seed, torch.float32, std)
