"""Growable, trimmable quantised KV cache (oracle side).

Page "sparkle mlx_streaming/core/cache/quant_kv.py", class
`AsymmetricQuantizedKVCache`: `step = 256`, `update_and_fetch`, `trim`,
`nbytes`, `state` / `meta_state`; page "sparkle mlx_streaming/mtp/kv_cache.py":
`commit_verified_prefix` (its trim branch), `_snapshot` / `_restore`,
`tile_caches` / `commit_tree_row`.

Readings:

* One length per sequence (`lens[b]`) instead of the page's single `offset`;
  the page's case is the one where every length is equal.  A speculative
  verify step accepts a different prefix per sequence, which needs this.
* Capacity grows by ceil(n/256)*256 tokens when an append would overflow and
  always stays a multiple of 256 (the page's slice-to-offset quirk before
  growing only changes `nbytes`).
* Rows at or past `lens[b]` are stale; nothing may read them.
* `dtype` "bf16" or "f32" is the input dtype (page `_init_quant(..., dt)`):
  scales and biases are bfloat16 or float32 values, and `append` takes M_b or
  the float32 blocks of M accordingly.
"""
from __future__ import annotations

import copy

import numpy as np

from . import codec

STEP = 256


class OracleCache:
    def __init__(self, batch: int, kv_heads: int, head_dim: int = 256, group_size: int = 64,
                 k_bits: int = 4, v_bits: int = 3, dtype: str = "bf16"):
        if dtype not in ("bf16", "f32"):
            raise ValueError("dtype must be 'bf16' or 'f32'")
        self.batch, self.kv_heads, self.head_dim = batch, kv_heads, head_dim
        self.group_size, self.k_bits, self.v_bits = group_size, k_bits, v_bits
        self.dtype = dtype
        self.capacity = 0
        self.lens = np.zeros(batch, dtype=np.int64)
        self.k = self.v = None

    def _alloc(self, cap):
        B, H, D, gs = self.batch, self.kv_heads, self.head_dim, self.group_size

        def triple(bits):
            return [np.zeros((B, H, cap, codec.packed_words(D, bits)), np.uint32),
                    np.zeros((B, H, cap, D // gs), np.float32),
                    np.zeros((B, H, cap, D // gs), np.float32)]
        return triple(self.k_bits), triple(self.v_bits)

    def _grow_for(self, n):
        need = int(self.lens.max()) + n
        if self.k is not None and need <= self.capacity:
            return
        new_cap = self.capacity + (STEP + n - 1) // STEP * STEP
        while new_cap < need:
            new_cap += STEP
        k, v = self._alloc(new_cap)
        if self.k is not None:
            for dst, src in zip(k + v, self.k + self.v):
                dst[:, :, :self.capacity] = src
        self.k, self.v, self.capacity = k, v, new_cap

    def append(self, keys, values, blocks):
        """Encode keys/values float32 [B, Hkv, n, D] and write rows [lens[b], lens[b]+n).

        blocks: M_b for a "bf16" cache, the float32 blocks of M for an "f32" one.
        """
        keys = np.asarray(keys, np.float32)
        values = np.asarray(values, np.float32)
        n = keys.shape[2]
        self._grow_for(n)
        kw, ks, kb = codec.encode_rows(keys, blocks, self.k_bits, self.group_size, self.dtype)
        vw, vs, vb = codec.encode_rows(values, blocks, self.v_bits, self.group_size, self.dtype)
        for b in range(self.batch):
            lo = int(self.lens[b])
            for dst, src in zip(self.k + self.v, (kw, ks, kb, vw, vs, vb)):
                dst[b, :, lo:lo + n] = src[b]
        self.lens += n

    def trim(self, n):
        """Per sequence: n = min(len, n); len -= n; return the trimmed counts (page `trim`)."""
        n = np.broadcast_to(np.asarray(n, dtype=np.int64), self.lens.shape)
        if (n < 0).any():
            raise ValueError("trim count must be non-negative")
        t = np.minimum(self.lens, n)
        self.lens = self.lens - t
        return t

    def nbytes(self) -> int:
        if self.k is None:
            return 0
        B, H, cap, D, gs = self.batch, self.kv_heads, self.capacity, self.head_dim, self.group_size
        words = codec.packed_words(D, self.k_bits) + codec.packed_words(D, self.v_bits)
        esz = 2 if self.dtype == "bf16" else 4
        return B * H * cap * (4 * words + esz * 4 * (D // gs))

    def dequantized(self, b: int, h: int):
        """(k_hat, v_hat) float64 [len, D] of rows [0, lens[b]) of slice (b, h)."""
        L, D, gs = int(self.lens[b]), self.head_dim, self.group_size
        kc = codec.unpack(self.k[0][b, h, :L], self.k_bits, D)
        vc = codec.unpack(self.v[0][b, h, :L], self.v_bits, D)
        kh = codec.dequantize(kc, self.k[1][b, h, :L], self.k[2][b, h, :L], gs)
        vh = codec.dequantize(vc, self.v[1][b, h, :L], self.v[2][b, h, :L], gs)
        return kh, vh

    def snapshot(self):
        """Deep copy of rows [0, len) plus lengths (page `_snapshot`: no aliasing)."""
        return copy.deepcopy((self.lens, self.capacity, self.k, self.v))

    def restore(self, snap):
        """Install a copy of a snapshot (page `_restore`: the snapshot stays intact)."""
        self.lens, self.capacity, self.k, self.v = copy.deepcopy(snap)

    def tile(self, paths: int):
        """Batch-1 cache -> batch-P cache with P copies (page `tile_caches`)."""
        if self.batch != 1:
            raise ValueError("tile needs a batch-1 cache")
        self.batch = paths
        self.lens = np.repeat(self.lens, paths)
        if self.k is not None:
            self.k = [np.repeat(a, paths, axis=0) for a in self.k]
            self.v = [np.repeat(a, paths, axis=0) for a in self.v]

    def keep_row(self, row: int):
        """Batch-P cache -> batch-1 cache holding sequence `row` (page `commit_tree_row`)."""
        self.batch = 1
        self.lens = self.lens[row:row + 1].copy()
        if self.k is not None:
            self.k = [a[row:row + 1].copy() for a in self.k]
            self.v = [a[row:row + 1].copy() for a in self.v]


def commit_verified_prefix(cache: OracleCache, verified_len: int, accepted_len) -> np.ndarray:
    """Trim the rejected suffix verified_len - accepted_len (per sequence).

    Raises ValueError when accepted_len exceeds verified_len, as the page does.
    """
    acc = np.asarray(accepted_len, dtype=np.int64)
    rejected = verified_len - acc
    if (rejected < 0).any():
        raise ValueError("accepted_len cannot exceed verified_len")
    return cache.trim(np.broadcast_to(rejected, cache.lens.shape))


def commit_verified_snapshot(cache: OracleCache, snapshots, accepted_len: int, verified_len=None) -> bool:
    """Page "kv_cache.py", `commit_verified_snapshot`: roll the cache back to the
    snapshot taken after `accepted_len` verified tokens.

    Its four branches, in the page's order: every verified token accepted
    (accepted_len == verified_len, when given) keeps the cache and returns True;
    accepted_len <= 0 returns False; accepted_len beyond the snapshots taken
    returns False; otherwise snapshot accepted_len - 1 is restored (a copy: the
    snapshot stays intact) and True is returned.
    """
    if verified_len is not None and accepted_len == verified_len:
        return True
    if accepted_len <= 0 or accepted_len > len(snapshots):
        return False
    cache.restore(snapshots[accepted_len - 1])
    return True
