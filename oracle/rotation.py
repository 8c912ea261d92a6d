"""Seed-fixed block-diagonal SO(4) rotation (oracle side).

Follows the page "sparkle mlx_streaming/core/cache/quant_kv.py", section
"SO(4) block rotation": `_quat_left`, `_quat_right_conj`, `build_block_so4`.

Readings where the page leaves the arithmetic open:

* Normalisation: the page divides a float32 quaternion by `np.linalg.norm` of
  it, in float32.  Read as: sum of squares accumulated in float32 in index
  order ((v0*v0 + v1*v1) + v2*v2) + v3*v3, each product and sum rounded to
  float32, a correctly rounded float32 square root, then an IEEE float32
  division of each component.
* Block product: `_quat_left(qL) @ _quat_right_conj(qR)` in float32 may differ
  by an ulp across BLAS builds.  Read as: each entry summed in float64 over the
  inner index k = 0..3 in order (float32 x float32 products are exact in
  float64), rounded once to float32.
* The matrices are taken exactly as printed.  The printed "right-conjugate"
  matrix is the transpose of the left-multiplication matrix, i.e. the
  left-multiplication matrix of conj(q); every block is therefore the
  left-multiplication matrix of qL * conj(qR).  It is orthogonal with
  determinant +1, which is all the method relies on.

The rotation is applied as a row vector times the matrix (`x @ M`), so only
the 64 diagonal 4x4 blocks are ever needed.
"""
from __future__ import annotations

import numpy as np

from .bf16 import round_bf16


def quat_left(q) -> np.ndarray:
    """4x4 matrix of v -> q * v (Hamilton product), as printed on the page."""
    w, x, y, z = (float(c) for c in q)
    return np.array([[w, -x, -y, -z],
                     [x, w, -z, y],
                     [y, z, w, -x],
                     [z, -y, x, w]], dtype=np.float64)


def quat_right_conj(q) -> np.ndarray:
    """The page's "right-multiply-by-conjugate" 4x4 matrix, as printed."""
    w, x, y, z = (float(c) for c in q)
    return np.array([[w, x, y, z],
                     [-x, w, z, -y],
                     [-y, -z, w, x],
                     [-z, y, -x, w]], dtype=np.float64)


def normalize_f32(v) -> np.ndarray:
    """float32 quaternion divided by its float32 Euclidean norm (reading above)."""
    v = np.asarray(v, dtype=np.float32)
    acc = np.float32(v[0] * v[0])
    for i in range(1, 4):
        acc = np.float32(acc + np.float32(v[i] * v[i]))
    norm = np.float32(np.sqrt(acc))
    return np.array([np.float32(v[i] / norm) for i in range(4)], dtype=np.float32)


def block_product(left: np.ndarray, right: np.ndarray) -> np.ndarray:
    """left @ right for 4x4 float64 matrices of float32 values, ordered sum, one rounding to f32."""
    out = np.empty((4, 4), dtype=np.float32)
    for i in range(4):
        for j in range(4):
            acc = 0.0
            for k in range(4):
                acc = acc + left[i, k] * right[k, j]
            out[i, j] = np.float32(acc)
    return out


def build_blocks(draws: np.ndarray) -> np.ndarray:
    """Rotation blocks float32 [D/4, 4, 4] from raw draws float32 [D/4, 2, 4]."""
    draws = np.asarray(draws, dtype=np.float32)
    nb = draws.shape[0]
    blocks = np.empty((nb, 4, 4), dtype=np.float32)
    for b in range(nb):
        ql = normalize_f32(draws[b, 0])
        qr = normalize_f32(draws[b, 1])
        blocks[b] = block_product(quat_left(ql), quat_right_conj(qr))
    return blocks


def blocks_bf16(blocks: np.ndarray) -> np.ndarray:
    """M_b: the blocks rounded to bfloat16 (returned as float32 values).

    `rotate_last` on the page casts the rotation to the activation dtype
    (`R.astype(x.dtype)`), bfloat16 here.
    """
    return round_bf16(np.asarray(blocks, dtype=np.float32))


def dense(blocks: np.ndarray) -> np.ndarray:
    """The full D x D block-diagonal matrix (tests only), float64."""
    nb = blocks.shape[0]
    m = np.zeros((4 * nb, 4 * nb), dtype=np.float64)
    for b in range(nb):
        m[4 * b:4 * b + 4, 4 * b:4 * b + 4] = blocks[b]
    return m
