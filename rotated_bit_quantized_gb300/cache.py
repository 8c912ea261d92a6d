"""Python face of libiqkv: rotation, quantised KV cache, attention.

Argument marshalling over the C ABI only: every step of the path runs in the
library's CUDA kernels.  Device memory comes from PyTorch (the caller's
allocator); work is enqueued on PyTorch's current CUDA stream.

Mirrors the page "sparkle mlx_streaming/core/cache/quant_kv.py"
(`build_block_so4`, `AsymmetricQuantizedKVCache.update_and_fetch`, `trim`,
`nbytes`, `state`, `meta_state`, `asym_quantized_sdpa`) and the page
"sparkle mlx_streaming/mtp/kv_cache.py" (`commit_verified_prefix`,
`_snapshot`/`_restore`, `commit_verified_snapshot`, `tile_caches`,
`commit_tree_row`).
"""
from __future__ import annotations

import ctypes
import math

import numpy as np
import torch

import seeded_inputs

from . import _abi
from ._abi import IQ_STEP, IQCacheDesc, check, lib


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(device_index: int | None = None) -> ctypes.c_void_p:
    """The current PyTorch stream of the device (the current device by default)."""
    if _raw_stream is not None:
        return ctypes.c_void_p(_raw_stream(torch.cuda.current_device() if device_index is None else device_index))
    return ctypes.c_void_p(torch.cuda.current_stream(device_index).cuda_stream)


class _OnDevice:
    """Make `index` the current device for a call, switching only when it is not."""

    __slots__ = ("index", "prev")

    def __init__(self, index: int):
        self.index, self.prev = index, None

    def __enter__(self):
        cur = torch.cuda.current_device()
        if cur != self.index:
            self.prev = cur
            torch.cuda.set_device(self.index)
        return self

    def __exit__(self, *exc):
        if self.prev is not None:
            torch.cuda.set_device(self.prev)
            self.prev = None


def _ptr(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def _need_cuda(t: torch.Tensor, dtype, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")
    return t.contiguous()


class Rotation:
    """Block-diagonal SO(4) rotation on the device (page `build_block_so4`).

    `blocks_f32` [D/4, 4, 4] float32 and `blocks_bf16` [D/4, 4, 4] bfloat16
    (M_b, what the cache and attention use).  The random draws come from
    ``numpy.random.default_rng(seed)`` in the page's order; the library
    normalises them and forms the blocks.
    """

    def __init__(self, seed: int = 0, head_dim: int = 256, device=None):
        device = torch.device(device or "cuda")
        nb = head_dim // 4
        self.seed, self.head_dim = seed, head_dim
        self.blocks_f32 = torch.empty((nb, 4, 4), dtype=torch.float32, device=device)
        self.blocks_bf16 = torch.empty((nb, 4, 4), dtype=torch.bfloat16, device=device)
        draws = np.ascontiguousarray(seeded_inputs.rotation_draws(seed, head_dim), dtype=np.float32)
        with torch.cuda.device(device):
            check(lib().iq_build_rotation(head_dim, draws.ctypes.data_as(ctypes.c_void_p),
                                          _ptr(self.blocks_f32), _ptr(self.blocks_bf16), _stream()),
                  "iq_build_rotation")


_DTYPE_CODES = {torch.bfloat16: _abi.IQ_DTYPE_BF16, torch.float32: _abi.IQ_DTYPE_F32}


class IQCache:
    """Rotated K4/V3 bit-packed KV cache with one length per sequence.

    Buffers follow the page's `(wq, scales, biases)` triples for keys and
    values; `lens` (host int32 [B]) is the authoritative length of each
    sequence.  Capacity grows in steps of 256 tokens, copying rows [0, len).
    `dtype` (bfloat16 or float32) is the dtype of the keys, values and
    queries the cache takes and of its scales and biases (the page's
    `_init_quant` stores them in the keys' dtype); a float32 cache rotates
    with the float32 blocks of M, a bfloat16 one with M_b.
    """

    BUFFERS = ("k_codes", "k_scales", "k_biases", "v_codes", "v_scales", "v_biases")

    def __init__(self, batch: int, kv_heads: int, head_dim: int = 256, group_size: int = 64,
                 k_bits: int = 4, v_bits: int = 3, capacity: int = IQ_STEP, device=None,
                 dtype=torch.bfloat16):
        if dtype not in _DTYPE_CODES:
            raise ValueError("dtype must be torch.bfloat16 or torch.float32")
        self.batch, self.kv_heads, self.head_dim = batch, kv_heads, head_dim
        self.group_size, self.k_bits, self.v_bits = group_size, k_bits, v_bits
        self.dtype = dtype
        self.device = torch.device(device or "cuda")
        if self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self._on = _OnDevice(self.device.index)
        self.lens = np.zeros(batch, dtype=np.int32)
        self._workspace = None
        self._ws_need = {}
        self._alloc(capacity)
        # bind the buffers through the library (validates them, zeroes the lengths)
        d = IQCacheDesc()
        bufs = (ctypes.c_void_p * 6)(*[getattr(self, n).data_ptr() for n in self.BUFFERS])
        check(lib().iq_cache_alloc(ctypes.byref(d), batch, kv_heads, head_dim, group_size, k_bits, v_bits,
                                   capacity, _DTYPE_CODES[dtype], bufs,
                                   self.lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))),
              "iq_cache_alloc")
        self._desc, self._desc_lens = d, self.lens

    # ---------------------------------------------------------------- storage
    def _alloc(self, capacity: int):
        sizes = (ctypes.c_size_t * 6)()
        check(lib().iq_cache_bytes(self.batch, self.kv_heads, self.head_dim, self.group_size,
                                   self.k_bits, self.v_bits, capacity, _DTYPE_CODES[self.dtype], sizes),
              "iq_cache_bytes")
        B, H = self.batch, self.kv_heads
        dev = self.device
        kw, vw = self.head_dim * self.k_bits // 32, self.head_dim * self.v_bits // 32
        ng = self.head_dim // self.group_size
        self.k_codes = torch.empty((B, H, capacity, kw), dtype=torch.int32, device=dev)
        self.k_scales = torch.empty((B, H, capacity, ng), dtype=self.dtype, device=dev)
        self.k_biases = torch.empty((B, H, capacity, ng), dtype=self.dtype, device=dev)
        self.v_codes = torch.empty((B, H, capacity, vw), dtype=torch.int32, device=dev)
        self.v_scales = torch.empty((B, H, capacity, ng), dtype=self.dtype, device=dev)
        self.v_biases = torch.empty((B, H, capacity, ng), dtype=self.dtype, device=dev)
        for name, n in zip(self.BUFFERS, sizes):
            assert getattr(self, name).numel() * getattr(self, name).element_size() == n
        self.capacity = capacity
        self._desc, self._desc_lens = None, None
        self._ws_need = {}

    def desc(self) -> IQCacheDesc:
        """The C descriptor of this cache (built once per allocation and lengths array;
        the library updates `lens` through it)."""
        d = self._desc
        if d is None or self._desc_lens is not self.lens:
            d = IQCacheDesc(self.batch, self.kv_heads, self.head_dim, self.group_size, self.k_bits,
                            self.v_bits, self.capacity, _DTYPE_CODES[self.dtype])
            for name in self.BUFFERS:
                setattr(d, name, getattr(self, name).data_ptr())
            if self.lens.dtype != np.int32 or not self.lens.flags["C_CONTIGUOUS"]:
                raise ValueError("lens must be a contiguous int32 array")
            d.lens = self.lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
            self._desc, self._desc_lens = d, self.lens
        return d

    @property
    def offset(self) -> int:
        """The page's single offset: defined when every sequence has the same length."""
        if not (self.lens == self.lens[0]).all():
            raise ValueError("sequences have different lengths; use .lens")
        return int(self.lens[0])

    @property
    def nbytes(self) -> int:
        d = self.desc()
        return int(lib().iq_cache_nbytes(ctypes.byref(d)))

    @property
    def state(self):
        """(keys, values), each the (codes, scales, biases) triple [B, Hkv, n, ...]
        of rows [0, n), n = the longest sequence (page `state`: the buffers
        sliced to the offset).  The tensors are copies, so later writes to the
        cache never change them."""
        n = int(self.lens.max()) if self.batch else 0

        def cut(t):
            return t[:, :, :n].clone()
        return ((cut(self.k_codes), cut(self.k_scales), cut(self.k_biases)),
                (cut(self.v_codes), cut(self.v_scales), cut(self.v_biases)))

    @state.setter
    def state(self, v) -> None:
        """Install (keys, values) triples of n rows: every sequence's length
        becomes n (page `state` setter: the offset becomes the arrays' length).
        The bit widths and group size follow the arrays' shapes, as the page's
        `meta_state` labels them, and the dtype follows the scales' dtype."""
        (kc, ks, kb), (vc, vs, vb) = v
        B, H, n = kc.shape[0], kc.shape[1], kc.shape[2]
        if (B, H) != (self.batch, self.kv_heads):
            raise ValueError("state batch / kv heads differ from the cache's")
        k_bits, v_bits = kc.shape[3] * 32 // self.head_dim, vc.shape[3] * 32 // self.head_dim
        group = self.head_dim // ks.shape[3]
        dtype = ks.dtype
        if dtype not in _DTYPE_CODES:
            raise ValueError(f"state scales have dtype {dtype}; bfloat16 or float32 expected")
        for t, name in zip((kc, ks, kb, vc, vs, vb), self.BUFFERS):
            want = torch.int32 if name.endswith("codes") else dtype
            if t.dtype != want or t.shape[:3] != (B, H, n):
                raise ValueError(f"state tensor for {name} has dtype {t.dtype} / shape {tuple(t.shape)}")
        if (k_bits, v_bits, group, dtype) != (self.k_bits, self.v_bits, self.group_size, self.dtype):
            self.k_bits, self.v_bits, self.group_size, self.dtype = k_bits, v_bits, group, dtype
            self.lens[:] = 0
            self._workspace = None
            self._alloc(max(IQ_STEP, int(math.ceil(max(n, 1) / IQ_STEP) * IQ_STEP)))
        self.reserve(n)
        for t, name in zip((kc, ks, kb, vc, vs, vb), self.BUFFERS):
            getattr(self, name)[:, :, :n].copy_(t.to(self.device))
        self.lens[:] = n

    @property
    def meta_state(self):
        """(group_size, k_bits, v_bits) as strings (page `meta_state`)."""
        return str(self.group_size), str(self.k_bits), str(self.v_bits)

    @meta_state.setter
    def meta_state(self, v) -> None:
        """The page's setter takes the labels of arrays installed by `state`; here
        the format is already fixed by those arrays, so the labels must agree."""
        gs, kb, vb = (int(x) for x in v)
        if (gs, kb, vb) != (self.group_size, self.k_bits, self.v_bits):
            raise ValueError(f"meta_state {v} disagrees with the cache's format "
                             f"({self.group_size}, {self.k_bits}, {self.v_bits})")

    def _fresh(self, batch: int, capacity: int) -> "IQCache":
        return IQCache(batch, self.kv_heads, self.head_dim, self.group_size, self.k_bits,
                       self.v_bits, capacity, self.device, self.dtype)

    def _gather_from(self, src: "IQCache", src_of) -> None:
        m = np.ascontiguousarray(src_of, dtype=np.int32)
        ds, dd = src.desc(), self.desc()
        with self._on:
            check(lib().iq_cache_gather(ctypes.byref(ds), ctypes.byref(dd),
                                        m.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                        _stream(self.device.index)),
                  "iq_cache_gather")
        self.lens[:] = np.ctypeslib.as_array(dd.lens, shape=(self.batch,))

    def reserve(self, capacity: int) -> None:
        """Grow to at least `capacity` tokens (multiple of 256), keeping rows [0, len)."""
        if capacity <= self.capacity:
            return
        new_cap = int(math.ceil(capacity / IQ_STEP) * IQ_STEP)
        old = IQCache.__new__(IQCache)
        old.__dict__.update(self.__dict__)
        old.lens = self.lens.copy()
        old._desc = None
        self._alloc(new_cap)
        ds, dd = old.desc(), self.desc()
        with self._on:
            check(lib().iq_cache_grow(ctypes.byref(ds), ctypes.byref(dd), _stream(self.device.index)),
                  "iq_cache_grow")

    def _rot(self, rotation: Rotation) -> ctypes.c_void_p:
        """The rotation blocks in the cache's dtype (the page's `R.astype(x.dtype)`)."""
        return _ptr(rotation.blocks_f32 if self.dtype == torch.float32 else rotation.blocks_bf16)

    # ---------------------------------------------------------------- page API
    def append(self, keys: torch.Tensor, values: torch.Tensor, rotation: Rotation) -> None:
        """Rotate, quantise, pack and append n tokens per sequence (page `update_and_fetch`).

        keys, values: CUDA tensors [B, Hkv, n, D] of the cache's dtype, unrotated.
        """
        keys = _need_cuda(keys, self.dtype, "keys")
        values = _need_cuda(values, self.dtype, "values")
        n = keys.shape[2]
        if tuple(keys.shape) != (self.batch, self.kv_heads, n, self.head_dim) or values.shape != keys.shape:
            raise ValueError("keys/values must be [B, Hkv, n, D]")
        need = int(self.lens.max()) + n
        if need > self.capacity:  # grow by ceil(n/256)*256 like the page, or more if needed
            self.reserve(max(need, self.capacity + int(math.ceil(n / IQ_STEP)) * IQ_STEP))
        d = self.desc()
        with self._on:
            check(lib().iq_cache_append(ctypes.byref(d), _ptr(keys), _ptr(values), n,
                                        self._rot(rotation), _stream(self.device.index)),
                  "iq_cache_append")

    def trim(self, n) -> np.ndarray:
        """Drop up to n tokens from each sequence; returns the counts dropped (page `trim`)."""
        counts = np.ascontiguousarray(np.broadcast_to(np.asarray(n, dtype=np.int32), (self.batch,)))
        out = np.zeros(self.batch, dtype=np.int32)
        d = self.desc()
        check(lib().iq_cache_trim(ctypes.byref(d), counts.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                  out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))), "iq_cache_trim")
        return out

    def workspace_bytes(self, q_heads: int, n_queries: int) -> int:
        """Workspace bytes iq_attend needs for this cache's batch (independent of the lengths)."""
        key = (self.batch, self.kv_heads, q_heads, n_queries)
        nb = self._ws_need.get(key)
        if nb is None:
            c = ctypes.c_size_t()
            d = self.desc()
            with self._on:
                check(lib().iq_attend_workspace(ctypes.byref(d), q_heads, n_queries, ctypes.byref(c)),
                      "iq_attend_workspace")
            nb = self._ws_need[key] = c.value
        return nb

    def attend(self, q: torch.Tensor, rotation: Rotation, causal: bool = False, scale: float | None = None,
               out: torch.Tensor | None = None, out_dtype=None,
               mask: torch.Tensor | None = None) -> torch.Tensor:
        """Attention of q [B, Hq, L, D] (the cache's dtype, unrotated) over the cache
        (page `asym_quantized_sdpa`).  The output is bf16 or float32 (`out_dtype`,
        default the cache's dtype, as the page returns the queries' dtype).

        mask: optional CUDA tensor [B, L, S] (S >= every length), shared by the
        heads: bool (keep where True) or float32 (added to the scores); not
        together with causal.  Returns [B, Hq, L, D] in unrotated space (the
        inverse rotation applied).
        """
        if mask is not None:
            return self._attend_mask(q, rotation, mask, causal, scale, out, out_dtype)
        q = _need_cuda(q, self.dtype, "q")
        B, Hq, L, D = q.shape
        if B != self.batch or D != self.head_dim:
            raise ValueError("q must be [B, Hq, L, D] matching the cache")
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        if out is None:
            out = torch.empty((B, Hq, L, D), dtype=out_dtype or self.dtype, device=q.device)
        out_f32 = 1 if out.dtype == torch.float32 else 0
        if out.dtype not in (torch.float32, torch.bfloat16) or not out.is_contiguous():
            raise ValueError("out must be a contiguous bf16 or f32 tensor")
        need = self.workspace_bytes(Hq, L)
        if self._workspace is None or self._workspace.numel() < need:
            # zeroed once: the status word at its head starts clear (iq_read_status clears it again)
            self._workspace = torch.zeros(max(need, 1 << 20), dtype=torch.uint8, device=self.device)
        d = self.desc()
        with self._on:
            check(lib().iq_attend(ctypes.byref(d), _ptr(q), Hq, L, float(scale), 1 if causal else 0,
                                  self._rot(rotation), _ptr(out), out_f32, _ptr(self._workspace),
                                  self._workspace.numel(), _stream(self.device.index)), "iq_attend")
        return out

    def _attend_mask(self, q, rotation, mask, causal, scale, out, out_dtype):
        if causal:
            raise ValueError("give either causal or an explicit mask")
        q = _need_cuda(q, self.dtype, "q")
        B, Hq, L, D = q.shape
        if B != self.batch or D != self.head_dim:
            raise ValueError("q must be [B, Hq, L, D] matching the cache")
        if not mask.is_cuda or mask.dim() != 3 or mask.shape[0] != B or mask.shape[1] != L:
            raise ValueError("mask must be a CUDA tensor [B, L, S]")
        if mask.dtype == torch.bool:
            kind = _abi.IQ_MASK_BOOL_U8
        elif mask.dtype == torch.float32:
            kind = _abi.IQ_MASK_ADD_F32
        else:
            raise ValueError("mask must be bool or float32")
        S = mask.shape[2]
        if S % 128 or not mask.is_contiguous():  # the library streams mask rows in 128-key pieces
            padded = torch.zeros((B, L, (S + 127) // 128 * 128), dtype=mask.dtype, device=mask.device)
            padded[:, :, :S] = mask
            mask = padded
        if kind == _abi.IQ_MASK_BOOL_U8:
            mask = mask.view(torch.uint8)
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        if out is None:
            out = torch.empty((B, Hq, L, D), dtype=out_dtype or self.dtype, device=q.device)
        if out.dtype not in (torch.float32, torch.bfloat16) or not out.is_contiguous():
            raise ValueError("out must be a contiguous bf16 or f32 tensor")
        need = self.workspace_bytes(Hq, L)
        if self._workspace is None or self._workspace.numel() < need:
            self._workspace = torch.zeros(max(need, 1 << 20), dtype=torch.uint8, device=self.device)
        d = self.desc()
        with self._on:
            check(lib().iq_attend_mask(ctypes.byref(d), _ptr(q), Hq, L, float(scale), kind, _ptr(mask),
                                       mask.shape[2], self._rot(rotation), _ptr(out),
                                       1 if out.dtype == torch.float32 else 0, _ptr(self._workspace),
                                       self._workspace.numel(), _stream(self.device.index)), "iq_attend_mask")
        return out

    def append_attend(self, keys: torch.Tensor, values: torch.Tensor, q: torch.Tensor, rotation: Rotation,
                      causal: bool = False, scale: float | None = None, out: torch.Tensor | None = None,
                      out_dtype=None) -> torch.Tensor:
        """`append(keys, values)` then `attend(q)` in one library call (the page's
        `update_and_fetch` followed by `asym_quantized_sdpa`): one kernel launch
        for decode-shaped steps, the same results as the two calls."""
        keys = _need_cuda(keys, self.dtype, "keys")
        values = _need_cuda(values, self.dtype, "values")
        q = _need_cuda(q, self.dtype, "q")
        n = keys.shape[2]
        if tuple(keys.shape) != (self.batch, self.kv_heads, n, self.head_dim) or values.shape != keys.shape:
            raise ValueError("keys/values must be [B, Hkv, n, D]")
        B, Hq, L, D = q.shape
        if B != self.batch or D != self.head_dim:
            raise ValueError("q must be [B, Hq, L, D] matching the cache")
        need = int(self.lens.max()) + n
        if need > self.capacity:
            self.reserve(max(need, self.capacity + int(math.ceil(n / IQ_STEP)) * IQ_STEP))
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        if out is None:
            out = torch.empty((B, Hq, L, D), dtype=out_dtype or self.dtype, device=q.device)
        if out.dtype not in (torch.float32, torch.bfloat16) or not out.is_contiguous():
            raise ValueError("out must be a contiguous bf16 or f32 tensor")
        out_f32 = 1 if out.dtype == torch.float32 else 0
        need_ws = self.workspace_bytes(Hq, L)
        if self._workspace is None or self._workspace.numel() < need_ws:
            self._workspace = torch.zeros(max(need_ws, 1 << 20), dtype=torch.uint8, device=self.device)
        d = self.desc()
        with self._on:
            check(lib().iq_cache_append_attend(ctypes.byref(d), _ptr(keys), _ptr(values), n, _ptr(q), Hq, L,
                                               float(scale), 1 if causal else 0, self._rot(rotation),
                                               _ptr(out), out_f32, _ptr(self._workspace), self._workspace.numel(),
                                               _stream(self.device.index)), "iq_cache_append_attend")
        return out

    def device_status(self) -> int:
        """Synchronise and return the kernels' status word (0 = all normal)."""
        if self._workspace is None:
            return 0
        st = ctypes.c_int()
        with self._on:
            code = lib().iq_read_status(_ptr(self._workspace), _stream(self.device.index), ctypes.byref(st))
        if code not in (_abi.IQ_OK, _abi.IQ_ERR_DEVICE):
            check(code, "iq_read_status")
        return st.value

    # ---------------------------------------------------------------- speculative decoding
    def commit_verified_prefix(self, verified_len: int, accepted_len) -> np.ndarray:
        """Trim the rejected suffix, verified_len - accepted_len per sequence
        (page "kv_cache.py", `commit_verified_prefix`, trimmable-cache branch)."""
        acc = np.broadcast_to(np.asarray(accepted_len, dtype=np.int64), (self.batch,))
        rejected = verified_len - acc
        if (rejected < 0).any():
            raise ValueError("accepted_len cannot exceed verified_len")
        return self.trim(rejected.astype(np.int32))

    def snapshot(self) -> "IQCache":
        """Independent copy of rows [0, len) (page `_snapshot`; never aliases)."""
        cap = max(IQ_STEP, int(math.ceil(max(int(self.lens.max()), 1) / IQ_STEP) * IQ_STEP))
        snap = self._fresh(self.batch, cap)
        snap._gather_from(self, np.arange(self.batch))
        return snap

    def restore(self, snap: "IQCache") -> None:
        """Install a copy of `snap` (page `_restore`: the snapshot stays intact)."""
        if snap.batch != self.batch:
            raise ValueError("snapshot batch differs")
        self.reserve(int(snap.lens.max()))
        self._gather_from(snap, np.arange(self.batch))

    def tile(self, paths: int) -> None:
        """Batch-1 cache -> batch-P cache of P identical paths (page `tile_caches`)."""
        if self.batch != 1:
            raise ValueError("tile needs a batch-1 cache")
        src = IQCache.__new__(IQCache)
        src.__dict__.update(self.__dict__)
        src.lens = self.lens.copy()
        self.batch = paths
        self.lens = np.zeros(paths, dtype=np.int32)
        self._workspace = None
        self._alloc(src.capacity)
        self._gather_from(src, np.zeros(paths, dtype=np.int32))

    def keep_row(self, row: int) -> None:
        """Batch-P cache -> batch-1 cache holding path `row` (page `commit_tree_row`)."""
        src = IQCache.__new__(IQCache)
        src.__dict__.update(self.__dict__)
        src.lens = self.lens.copy()
        self.batch = 1
        self.lens = np.zeros(1, dtype=np.int32)
        self._workspace = None
        self._alloc(src.capacity)
        self._gather_from(src, np.array([row], dtype=np.int32))

    def commit_tree_row(self, verified_len: int, accepted_len: int, row: int) -> None:
        """Trim the rejected suffix of every path, then keep path `row` (page `commit_tree_row`)."""
        self.commit_verified_prefix(verified_len, accepted_len)
        self.keep_row(row)


def commit_verified_snapshot(cache: IQCache, snapshots, accepted_len: int,
                             verified_len: int | None = None) -> bool:
    """Restore the snapshot taken after `accepted_len` verified tokens
    (page "kv_cache.py", `commit_verified_snapshot`)."""
    if verified_len is not None and accepted_len == verified_len:
        return True
    if accepted_len <= 0 or accepted_len > len(snapshots):
        return False
    cache.restore(snapshots[accepted_len - 1])
    return True
