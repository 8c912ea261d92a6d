"""bfloat16 rounding from bit operations on float32 (no torch, no ml_dtypes).

bfloat16 keeps the top 16 bits of an IEEE float32.  Rounding is
round-to-nearest, ties to even, which is what both the page's MLX arrays
(`x.astype(bfloat16)`) and CUDA's `__float2bfloat16_rn` do.
"""
from __future__ import annotations

import numpy as np


def f32_to_bf16_bits(x) -> np.ndarray:
    """float32 values -> uint16 bfloat16 bit patterns, round to nearest even."""
    a = np.asarray(x, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    quiet = (u >> np.uint64(16)) | np.uint64(0x40)
    out = np.where(np.isnan(a), quiet, rounded) & np.uint64(0xFFFF)
    return out.astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """uint16 bfloat16 bit patterns -> float32 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def round_bf16(x) -> np.ndarray:
    """Round float32 values to the nearest bfloat16, returned as float32."""
    return bf16_bits_to_f32(f32_to_bf16_bits(x))


def ulp_bf16(x) -> np.ndarray:
    """Spacing of bfloat16 numbers at |x| (2^(e-7) for normal x)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)
