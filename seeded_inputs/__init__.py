"""Seeded synthetic inputs shared by the oracle, the tests and the benchmark.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no rotation, quantisation, packing or attention).  Both
the CPU oracle and the CUDA path consume what it returns, so the two sides see
bit-identical inputs without sharing any code that computes the method.

Recipe (stated once here, restated in the design notes):

* Rotation draws follow the page "sparkle mlx_streaming/core/cache/quant_kv.py",
  `build_block_so4`: one ``numpy.random.default_rng(seed)``; for every 4-wide
  block, four standard normals for the left quaternion, then four for the right
  one, each batch drawn in float64 and cast to float32.  Only the raw draws are
  returned; normalising them and building the blocks is the method's job.
* Token data is drawn per (sequence b, kv head h) slice from its own generator
  ``default_rng((data_seed, stream, ...))`` so that any slice can be rebuilt on
  its own.  Values are float32 standard normals (``dtype=float32`` ziggurat),
  rounded to bfloat16 by round-to-nearest-even (torch's conversion), or left
  as float32 draws when float32 data is asked for (``dtype=torch.float32``).  Keys of
  the outlier workloads get 8 distinct channels per (b, h), chosen with
  ``rng.choice(256, 8, replace=False)`` before any token is drawn, scaled by 20
  before rounding.  Decode/verify steps draw new tokens from a generator keyed
  by the step, reusing the slice's outlier channels.
* Speculative-verify acceptance counts: ``default_rng(50).integers(0, 5,
  size=(steps, B))``.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

STREAM_PREFILL = 1
STREAM_STEP = 2
STREAM_QUERY = 3
OUTLIER_CHANNELS = 8
OUTLIER_GAIN = 20.0

_POOL = None


def _pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=16)
    return _POOL


def rotation_draws(seed: int, head_dim: int, blocks_of: int = 4) -> np.ndarray:
    """Raw quaternion draws, float32 [head_dim/4, 2, 4] (left, right per block).

    Same generator calls, in the same order, as `build_block_so4` on the page
    "quant_kv.py": per block ``standard_normal(4).astype(float32)`` for the left
    quaternion and then for the right one.
    """
    if head_dim % blocks_of != 0:
        raise ValueError("head_dim must be a multiple of blocks_of")
    rng = np.random.default_rng(seed)
    nb = head_dim // blocks_of
    out = np.empty((nb, 2, blocks_of), dtype=np.float32)
    for b in range(nb):
        out[b, 0] = rng.standard_normal(blocks_of).astype(np.float32)
        out[b, 1] = rng.standard_normal(blocks_of).astype(np.float32)
    return out


def to_bf16(x: np.ndarray) -> torch.Tensor:
    """float32 numpy array -> CPU bfloat16 tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def _outliers(rng: np.random.Generator, head_dim: int) -> np.ndarray:
    return rng.choice(head_dim, OUTLIER_CHANNELS, replace=False)


def _slice_tokens(data_seed, b, h, n, head_dim, outliers, stream, step):
    if stream == STREAM_PREFILL:
        rng = np.random.default_rng((data_seed, STREAM_PREFILL, b, h))
        ch = _outliers(rng, head_dim) if outliers else None
    else:
        ch = outlier_channels(data_seed, b, h, head_dim) if outliers else None
        rng = np.random.default_rng((data_seed, STREAM_STEP, step, b, h))
    k = rng.standard_normal((n, head_dim), dtype=np.float32)
    v = rng.standard_normal((n, head_dim), dtype=np.float32)
    if ch is not None:
        k[:, ch] *= np.float32(OUTLIER_GAIN)
    return k, v


def outlier_channels(data_seed: int, b: int, h: int, head_dim: int = 256) -> np.ndarray:
    """The 8 outlier channels of slice (b, h): the first draw of its prefill generator."""
    rng = np.random.default_rng((data_seed, STREAM_PREFILL, b, h))
    return _outliers(rng, head_dim)


def _as(x: np.ndarray, dtype) -> torch.Tensor:
    if dtype == torch.float32:
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return to_bf16(x)


def kv_tokens(data_seed: int, batch: int, kv_heads: int, n: int, head_dim: int = 256,
              outliers: bool = False, step: int | None = None,
              slices: list[tuple[int, int]] | None = None, dtype=torch.bfloat16):
    """K and V tokens as CPU tensors [B, Hkv, n, D] (bfloat16, or the float32
    draws themselves for ``dtype=torch.float32``).

    ``step=None`` gives the prefill draw of every slice; ``step=s`` the tokens
    appended at decode/verify step ``s``.  ``slices`` restricts the draw to the
    listed (b, h) pairs (the others are left as zeros) so a checker can rebuild
    only what it samples.
    """
    stream = STREAM_PREFILL if step is None else STREAM_STEP
    k = torch.zeros((batch, kv_heads, n, head_dim), dtype=dtype)
    v = torch.zeros_like(k)
    todo = slices if slices is not None else [(b, h) for b in range(batch) for h in range(kv_heads)]

    def work(bh):
        b, h = bh
        kk, vv = _slice_tokens(data_seed, b, h, n, head_dim, outliers, stream, step)
        k[b, h] = _as(kk, dtype)
        v[b, h] = _as(vv, dtype)

    list(_pool().map(work, todo))
    return k, v


def kv_slice(data_seed: int, b: int, h: int, n: int, head_dim: int = 256,
             outliers: bool = False, step: int | None = None, dtype=torch.bfloat16):
    """K and V tokens of the single slice (b, h) as CPU tensors [n, D];
    identical to ``kv_tokens(...)[.][b, h]``."""
    stream = STREAM_PREFILL if step is None else STREAM_STEP
    k, v = _slice_tokens(data_seed, b, h, n, head_dim, outliers, stream, step)
    return _as(k, dtype), _as(v, dtype)


def queries(data_seed: int, batch: int, q_heads: int, n: int, head_dim: int = 256,
            step: int = 0, dtype=torch.bfloat16) -> torch.Tensor:
    """Queries as a CPU tensor [B, Hq, n, D], ~N(0, 1) (bfloat16, or float32 draws)."""
    out = torch.empty((batch, q_heads, n, head_dim), dtype=dtype)
    for b in range(batch):
        rng = np.random.default_rng((data_seed, STREAM_QUERY, step, b))
        out[b] = _as(rng.standard_normal((q_heads, n, head_dim), dtype=np.float32), dtype)
    return out


def accepted_lengths(steps: int, batch: int, draft: int = 4, seed: int = 50) -> np.ndarray:
    """Accepted prefix length per (step, sequence), uniform on 0..draft."""
    return np.random.default_rng(seed).integers(0, draft + 1, size=(steps, batch))


def garbage_like(shape, seed: int = 7) -> np.ndarray:
    """Random 32-bit words used to pre-fill buffers whose stale rows must never be read."""
    return np.random.default_rng(seed).integers(0, 2 ** 32, size=shape, dtype=np.uint32)


# The five workloads (sizes and seeds only).  `prefill` tokens are appended in
# one call; each of `steps` steps appends `append` tokens per sequence and then
# attends `queries` new queries per sequence (`causal` as stated).
WORKLOADS = {
    1: dict(name="tiny", B=1, Hq=1, Hkv=1, prefill=256, outliers=False, steps=0, append=0,
            queries=1, causal=False, seed=1),
    2: dict(name="single_stream_decode", B=1, Hq=16, Hkv=2, prefill=4096, outliers=True, steps=0,
            append=0, queries=1, causal=False, seed=2),
    3: dict(name="chunked_prefill", B=1, Hq=16, Hkv=2, prefill=0, outliers=True, steps=16,
            append=2048, queries=2048, causal=True, trim_after=1000, seed=3),
    4: dict(name="batched_decode", B=32, Hq=16, Hkv=2, prefill=32768, outliers=True, steps=64,
            append=1, queries=1, causal=True, seed=4),
    5: dict(name="spec_verify", B=8, Hq=16, Hkv=2, prefill=131072, outliers=True, steps=32,
            append=4, queries=4, causal=True, accept_seed=50, seed=5),
}
