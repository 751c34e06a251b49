"""Seeded synthetic inputs for the ternary (PQ2) x INT8 matmul.

This module holds only the data recipe: random draws and the byte layout of
the raw block format.  It does none of the method's arithmetic (no decode, no
quantisation, no dot products), so both the CUDA path and the CPU oracle can
consume what it produces.

Raw block format (page "Kernel experiments: recorded evidence", Test 1 and
Diagram 1): each row is K/128 blocks of 34 bytes; bytes 0-1 hold the block's
fp16 scale (little-endian), bytes 2..33 hold 32 code bytes, and weight k of
the block is stored in bits 2(k%4)..2(k%4)+1 of code byte k/4.

Workload recipe (the pages' synthetic setup, Tests 12 and 24: random codes,
fp16 scales overwritten with a small positive range):
  * codes iid uniform over {0, 1, 2} (so weights -1, 0, +1, zero fraction 1/3)
  * weight scales fp16 uniform in [0.005, 0.05]
  * activations bf16 N(0, 1); optionally a seeded 1% of the K channels, the
    same for every row, multiplied by 20 (outlier channels)
"""
from __future__ import annotations

import torch

GROUP = 128
BLOCK_BYTES = 34


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def raw_weights(N: int, K: int, seed: int, device="cpu", *,
                scale_lo: float = 0.005, scale_hi: float = 0.05,
                code_values: int = 3) -> torch.Tensor:
    """Raw PQ2 matrix u8[N][K/128*34].

    code_values=3 draws codes from {0,1,2} (ternary data); code_values=4 also
    draws code 3 (every packed byte value can occur, as in the pages' random
    byte fixtures)."""
    if K % GROUP:
        raise ValueError("K must be a multiple of 128")
    G = K // GROUP
    g = _gen(seed, device)
    codes = torch.randint(0, code_values, (N, G, 32, 4), generator=g,
                          device=device, dtype=torch.uint8)
    packed = (codes[..., 0] | (codes[..., 1] << 2) | (codes[..., 2] << 4)
              | (codes[..., 3] << 6))
    scales = (torch.rand((N, G), generator=g, device=device, dtype=torch.float32)
              * (scale_hi - scale_lo) + scale_lo).to(torch.float16)
    raw = torch.empty((N, G, BLOCK_BYTES), dtype=torch.uint8, device=device)
    raw[:, :, 0:2] = scales.view(torch.uint8).view(N, G, 2)
    raw[:, :, 2:] = packed
    return raw.view(N, G * BLOCK_BYTES)


PTQ_BLOCK_BYTES = 28


def ptq_raw_weights(N: int, K: int, seed: int, device="cpu", *,
                    scale_lo: float = 0.005, scale_hi: float = 0.05) -> torch.Tensor:
    """Raw PTQ1_0 matrix u8[N][K/128*28] (page "KERNEL_REPORT: PTQ1_0
    small-batch decoding on the PrismML fork, RTX 3060 12GB"): per block, 26
    trit bytes (24 qs, 2 qh) drawn uniformly over 0..255, then the fp16
    scale in bytes 26-27.  Every byte value is a valid five-trit word, so
    uniform bytes give each trit value with probability about 1/3."""
    if K % GROUP:
        raise ValueError("K must be a multiple of 128")
    G = K // GROUP
    g = _gen(seed, device)
    trit_bytes = torch.randint(0, 256, (N, G, 26), generator=g, device=device,
                               dtype=torch.int32).to(torch.uint8)
    scales = (torch.rand((N, G), generator=g, device=device, dtype=torch.float32)
              * (scale_hi - scale_lo) + scale_lo).to(torch.float16)
    raw = torch.empty((N, G, PTQ_BLOCK_BYTES), dtype=torch.uint8, device=device)
    raw[:, :, :26] = trit_bytes
    raw[:, :, 26:] = scales.view(torch.uint8).view(N, G, 2)
    return raw.view(N, G * PTQ_BLOCK_BYTES)


def activations(M: int, K: int, seed: int, device="cpu", *,
                dtype=torch.bfloat16, outlier_frac: float = 0.0,
                outlier_scale: float = 20.0) -> torch.Tensor:
    """Activations x[M][K] ~ N(0,1) in `dtype`; with outlier_frac > 0 a seeded
    subset of round(outlier_frac*K) channels (shared by all rows) is scaled."""
    g = _gen(seed, device)
    x = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    if outlier_frac > 0:
        n_out = max(1, int(round(outlier_frac * K)))
        idx = torch.randperm(K, generator=g, device=device)[:n_out]
        x[:, idx] *= outlier_scale
    return x.to(dtype)


def raw_from_parts(codes_0123: torch.Tensor, scale_bits: torch.Tensor) -> torch.Tensor:
    """Raw matrix from explicit codes u8[N][K] (values 0..3, weight k at field
    k%4 of byte k/4) and fp16 scale bit patterns i16/u16[N][K/128].
    Used for hand-built fixtures (worked example, special cases)."""
    N, K = codes_0123.shape
    G = K // GROUP
    c = codes_0123.to(torch.uint8).view(N, G, 32, 4)
    packed = c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)
    raw = torch.empty((N, G, BLOCK_BYTES), dtype=torch.uint8)
    sb = scale_bits.to(torch.int32)
    raw[:, :, 0] = (sb & 0xFF).to(torch.uint8)
    raw[:, :, 1] = ((sb >> 8) & 0xFF).to(torch.uint8)
    raw[:, :, 2:] = packed
    return raw.view(N, G * BLOCK_BYTES)


def bits_u16(x: torch.Tensor):
    """bf16/f16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
