"""Rotate, group-quantise, bit-pack (oracle side).

Page "sparkle mlx_streaming/core/cache/quant_kv.py": `rotate_last`,
`_packed_words`, the `(wq, scales, biases)` triple of
`AsymmetricQuantizedKVCache._init_quant`, and the two `mx.quantize` calls of
`update_and_fetch`.  The page does not print the quantiser; the affine
min/max rule used here is the one stated for the method: scale =
(max - min) / (2^b - 1), bias = min, code = clamp(round((x - bias)/scale)).

Readings:

* Rotation `x @ R.astype(bfloat16)` with bfloat16 x: each product
  x_i * M_b[i][j] is exact in float32; the four products of a 4-wide block are
  summed in float32 in order i = 0..3 and the sum is rounded once to bfloat16.
* Scales and biases are stored in the input dtype (bfloat16) as the page's
  `_init_quant(..., dt)` does: s_hat = bf16(scale) and b_hat = min (already a
  bfloat16 value).  Codes are computed from the stored s_hat and b_hat with a
  float32 subtraction, an IEEE float32 division and round-half-to-even.
  A constant group (s_hat == 0) gets all codes 0.
* Packing is a pure LSB-first bit stream per row: element i occupies stream
  bits [i*b, i*b + b); 32-bit word w holds stream bits [32w, 32w + 32).
  Rows hold dim*bits/32 words (`_packed_words`).
* float32 inputs (the page's `rotate_last` casts M to the input's dtype and
  `_init_quant` stores scales and biases in it): `x @ M` in float32 is read
  as a row vector times the 4x4 block taken in index order, every product
  and every partial sum rounded to float32, i.e.
  (((x0*M[0][j] + x1*M[1][j]) + x2*M[2][j]) + x3*M[3][j]) with no fused
  multiply-add; the scale is stored as computed (no bfloat16 rounding), the
  bias is the float32 minimum, and the codes come from them exactly as above.
"""
from __future__ import annotations

import numpy as np

from .bf16 import round_bf16


def packed_words(dim: int, bits: int) -> int:
    """uint32 words per packed row: dim*bits//32 (page `_packed_words`)."""
    return dim * bits // 32


def rotate(x, blocks_b) -> np.ndarray:
    """bf16(x @ M_b) per 4-wide block; x float32 [..., D] of bfloat16 values."""
    x = np.asarray(x, dtype=np.float32)
    m = np.asarray(blocks_b, dtype=np.float32)
    nb = m.shape[0]
    x4 = x.reshape(x.shape[:-1] + (nb, 4))
    acc = x4[..., 0, None] * m[:, 0, :]
    for i in range(1, 4):
        acc = (acc + x4[..., i, None] * m[:, i, :]).astype(np.float32)
    return round_bf16(acc.reshape(x.shape))


def rotate_f32(x, blocks) -> np.ndarray:
    """x @ M per 4-wide block for float32 x and the float32 blocks of M:
    products and sums rounded to float32 one at a time, in index order."""
    x = np.asarray(x, dtype=np.float32)
    m = np.asarray(blocks, dtype=np.float32)
    nb = m.shape[0]
    x4 = x.reshape(x.shape[:-1] + (nb, 4))
    acc = (x4[..., 0, None] * m[:, 0, :]).astype(np.float32)
    for i in range(1, 4):
        prod = (x4[..., i, None] * m[:, i, :]).astype(np.float32)
        acc = (acc + prod).astype(np.float32)
    return acc.reshape(x.shape)


def quantize(x, bits: int, group_size: int, meta: str = "bf16"):
    """Affine group quantisation of float32 rows [..., D].

    Returns (codes uint8 [..., D], s_hat float32 [..., D/gs], b_hat float32 [..., D/gs]).
    meta "bf16": the rows hold bfloat16 values and s_hat is the scale rounded
    to bfloat16; meta "f32": s_hat is the float32 scale itself.
    """
    if meta not in ("bf16", "f32"):
        raise ValueError("meta must be 'bf16' or 'f32'")
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[-1]
    g = x.reshape(x.shape[:-1] + (d // group_size, group_size))
    mn = g.min(axis=-1)
    mx = g.max(axis=-1)
    levels = np.float32(2 ** bits - 1)
    scale = ((mx - mn).astype(np.float32) / levels).astype(np.float32)
    s_hat = round_bf16(scale) if meta == "bf16" else scale
    b_hat = mn.astype(np.float32)
    diff = (g - b_hat[..., None]).astype(np.float32)
    safe = np.where(s_hat == 0, np.float32(1), s_hat).astype(np.float32)
    ratio = (diff / safe[..., None]).astype(np.float32)
    codes = np.clip(np.rint(ratio), 0, 2 ** bits - 1)
    codes = np.where((s_hat == 0)[..., None], 0, codes)
    return codes.reshape(x.shape).astype(np.uint8), s_hat, b_hat


def dequantize(codes, s_hat, b_hat, group_size: int) -> np.ndarray:
    """x_hat = s_hat * code + b_hat per group, in float64 (exact for these inputs)."""
    c = np.asarray(codes, dtype=np.float64)
    d = c.shape[-1]
    cg = c.reshape(c.shape[:-1] + (d // group_size, group_size))
    out = cg * np.asarray(s_hat, np.float64)[..., None] + np.asarray(b_hat, np.float64)[..., None]
    return out.reshape(c.shape)


def pack(codes, bits: int) -> np.ndarray:
    """LSB-first bit stream of b-bit codes [..., D] -> uint32 words [..., D*b/32]."""
    c = np.asarray(codes, dtype=np.uint64)
    d = c.shape[-1]
    nw = packed_words(d, bits)
    words = np.zeros(c.shape[:-1] + (nw,), dtype=np.uint64)
    mask32 = np.uint64(0xFFFFFFFF)
    for i in range(d):
        pos = i * bits
        w, s = divmod(pos, 32)
        words[..., w] |= (c[..., i] << np.uint64(s)) & mask32
        if s + bits > 32:
            words[..., w + 1] |= c[..., i] >> np.uint64(32 - s)
    return words.astype(np.uint32)


def unpack(words, bits: int, dim: int) -> np.ndarray:
    """Inverse of `pack`: uint32 words [..., D*b/32] -> codes uint8 [..., D]."""
    w = np.asarray(words, dtype=np.uint64)
    out = np.zeros(w.shape[:-1] + (dim,), dtype=np.uint64)
    mask = np.uint64(2 ** bits - 1)
    for i in range(dim):
        pos = i * bits
        k, s = divmod(pos, 32)
        v = w[..., k] >> np.uint64(s)
        if s + bits > 32:
            v = v | (w[..., k + 1] << np.uint64(32 - s))
        out[..., i] = v & mask
    return out.astype(np.uint8)


def encode_rows(x, blocks, bits: int, group_size: int, dtype: str = "bf16"):
    """One cache row per input row: rotate, quantise, pack.

    dtype "bf16": x holds bfloat16 values and `blocks` is M_b; dtype "f32": x is
    float32 and `blocks` the float32 blocks of M.
    Returns (words uint32 [..., D*b/32], s_hat f32 [..., D/gs], b_hat f32 [..., D/gs]).
    """
    xr = rotate(x, blocks) if dtype == "bf16" else rotate_f32(x, blocks)
    codes, s_hat, b_hat = quantize(xr, bits, group_size, meta=dtype)
    return pack(codes, bits), s_hat, b_hat
