"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and the bench.

This module holds no attention arithmetic. It draws N(0,1) values from a
seeded NumPy PCG64 stream (or, for inputs too large to draw on the host, a
seeded torch generator on the device), rounds fp32 draws to bfloat16 with
round-to-nearest-even, and hands out the same bits to both sides: the CUDA
path gets them as bf16 tensors, the oracle gets their exact fp64 upcast.

The workload shapes follow the benchmark setup of the page
"FlashAttention：快速且内存高效的准确注意力机制" (cloud.tencent.com.cn),
section "性能表现 / 加速效果": head dim 64 or 128, hidden 2048 (32 or 16
heads), sequence length 512..16k, batch = 16k / seqlen.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "bf16_bits_to_f64",
    "normal_bf16_bits",
    "alibi_slopes_geometric",
    "attention_inputs",
    "seed_for",
]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bits to float32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bits to float64."""
    return bf16_bits_to_f32(bits).astype(np.float64)


def normal_bf16_bits(shape, seed: int, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) draws: N(0,1) float32 from PCG64(seed), times std in float32,
    rounded once to bf16; returns uint16 bits."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x = x * np.float32(std)
    return f32_to_bf16_bits(x)


def alibi_slopes_geometric(H: int) -> np.ndarray:
    """The mask-variant workload's fp32 ALiBi slopes, 2^(-8(h+1)/H) for h = 0..H-1."""
    h = np.arange(H, dtype=np.float64)
    return np.exp2(-8.0 * (h + 1.0) / H).astype(np.float32)


def seed_for(config_id: int, variant: int) -> int:
    """Seed convention: 1000 * config id + variant index."""
    return 1000 * int(config_id) + int(variant)


def attention_inputs(B, Sq, Sk, H, D, seed, with_dout=False):
    """q (B,Sq,H,D), k, v (B,Sk,H,D) and optionally dO (B,Sq,H,D), all as bf16 bits.

    Each tensor has its own sub-seed so adding dO does not change q, k or v.
    """
    out = {
        "q": normal_bf16_bits((B, Sq, H, D), seed * 8 + 0),
        "k": normal_bf16_bits((B, Sk, H, D), seed * 8 + 1),
        "v": normal_bf16_bits((B, Sk, H, D), seed * 8 + 2),
    }
    if with_dout:
        out["dout"] = normal_bf16_bits((B, Sq, H, D), seed * 8 + 3)
    return out


def device_normal_bf16(shape, seed: int, device="cuda"):
    """Large inputs drawn directly on the device: torch N(0,1) fp32 from a seeded
    device generator, rounded to bf16 by torch's round-to-nearest-even cast.
    Used where a host draw would take minutes (multi-GB KV caches)."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    # Draw in slabs so the fp32 intermediate stays small.
    flat = out.view(-1)
    n = flat.numel()
    step = 1 << 28
    for s in range(0, n, step):
        e = min(n, s + step)
        flat[s:e].copy_(torch.randn(e - s, generator=g, device=device, dtype=torch.float32))
    return out
