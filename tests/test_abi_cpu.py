"""The C-ABI library loads, exports every symbol of include/iqkv.h, and rejects
bad arguments on the host before touching a device.  Runs without a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from rotated_bit_quantized_gb300 import build
    build.build()
    from rotated_bit_quantized_gb300 import _abi
    return _abi.lib()


def header_functions():
    text = open(os.path.join(ROOT, "include", "iqkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(iq_[a-z_0-9]+)\s*\(", text))


def test_every_declared_symbol_is_exported(L):
    declared = header_functions()
    from rotated_bit_quantized_gb300 import _abi
    assert declared == set(_abi.EXPORTS)
    for name in declared:
        assert hasattr(L, name), name


def test_status_strings(L):
    assert L.iq_status_string(0) == b"IQ_OK"
    assert L.iq_status_string(2) == b"IQ_ERR_CAPACITY"
    assert L.iq_status_string(99) == b"IQ_ERR_UNKNOWN"


def test_cache_bytes(L):
    out = (ctypes.c_size_t * 6)()
    assert L.iq_cache_bytes(2, 3, 256, 64, 4, 3, 512, 0, out) == 0
    rows = 2 * 3 * 512
    assert list(out) == [rows * 128, rows * 8, rows * 8, rows * 96, rows * 8, rows * 8]
    # float32 scales and biases (page `_init_quant(..., dt)` with float32 keys): 4 bytes per group
    assert L.iq_cache_bytes(2, 3, 256, 64, 4, 3, 512, 1, out) == 0
    assert list(out) == [rows * 128, rows * 16, rows * 16, rows * 96, rows * 16, rows * 16]
    assert L.iq_cache_bytes(2, 3, 256, 64, 4, 3, 512, 2, out) == 1     # unknown dtype
    assert L.iq_cache_bytes(2, 3, 256, 64, 4, 3, 500, 0, out) == 1     # not a multiple of 256
    assert L.iq_cache_bytes(2, 3, 128, 64, 4, 3, 512, 0, out) == 4     # other head_dim
    assert L.iq_cache_bytes(2, 3, 256, 64, 7, 3, 512, 0, out) == 4     # a width the page does not list
    assert L.iq_cache_bytes(2, 3, 256, 16, 4, 3, 512, 0, out) == 4     # group size not built
    assert L.iq_cache_bytes(300, 3, 256, 64, 4, 3, 512, 0, out) == 4   # batch above maximum
    assert b"256" in L.iq_last_error() or L.iq_last_error()


@pytest.mark.parametrize("kb,vb,gs", [(2, 2, 32), (3, 5, 128), (5, 6, 64), (8, 8, 128), (6, 3, 32)])
def test_cache_bytes_other_formats(L, kb, vb, gs):
    # page `_packed_words`: dim * bits / 32 words per row; one bf16 scale and
    # bias per group
    out = (ctypes.c_size_t * 6)()
    rows = 2 * 256
    ng = 256 // gs
    for dtype, esz in ((0, 2), (1, 4)):
        assert L.iq_cache_bytes(1, 2, 256, gs, kb, vb, 256, dtype, out) == 0
        assert list(out) == [rows * 8 * kb * 4, rows * ng * esz, rows * ng * esz, rows * 8 * vb * 4,
                             rows * ng * esz, rows * ng * esz]


def fake_desc(batch=2, cap=256, lens=(3, 4), align=0, dtype=0):
    from rotated_bit_quantized_gb300._abi import IQCacheDesc
    d = IQCacheDesc(batch, 2, 256, 64, 4, 3, cap, dtype)
    base = 0x10000000 + align
    for i, name in enumerate(("k_codes", "k_scales", "k_biases", "v_codes", "v_scales", "v_biases")):
        setattr(d, name, base + i * 0x1000000)
    arr = np.array(lens, dtype=np.int32)
    d.lens = arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    return d, arr


def test_check_and_trim_host_only(L):
    d, lens = fake_desc()
    assert L.iq_cache_check(ctypes.byref(d)) == 0
    d2, _ = fake_desc(align=4)
    assert L.iq_cache_check(ctypes.byref(d2)) == 1
    d3, _ = fake_desc(lens=(3, 300))
    assert L.iq_cache_check(ctypes.byref(d3)) == 1
    n = np.array([5, 1], dtype=np.int32)
    out = np.zeros(2, dtype=np.int32)
    P = ctypes.POINTER(ctypes.c_int32)
    assert L.iq_cache_trim(ctypes.byref(d), n.ctypes.data_as(P), out.ctypes.data_as(P)) == 0
    assert out.tolist() == [3, 1] and lens.tolist() == [0, 3]
    neg = np.array([-1, 0], dtype=np.int32)
    assert L.iq_cache_trim(ctypes.byref(d), neg.ctypes.data_as(P), out.ctypes.data_as(P)) == 1
    assert lens.tolist() == [0, 3]
    assert L.iq_cache_nbytes(ctypes.byref(d)) == 2 * 2 * 256 * 256
    df, _ = fake_desc(dtype=1)
    assert L.iq_cache_check(ctypes.byref(df)) == 0
    assert L.iq_cache_nbytes(ctypes.byref(df)) == 2 * 2 * 256 * (128 + 96 + 4 * 16)
    dx, _ = fake_desc(dtype=5)
    assert L.iq_cache_check(ctypes.byref(dx)) == 1


def test_append_and_attend_reject_before_launch(L):
    d, lens = fake_desc(lens=(250, 10))
    p = ctypes.c_void_p(0x20000000)
    # capacity: 250 + 7 > 256
    assert L.iq_cache_append(ctypes.byref(d), p, p, 7, p, None) == 2
    assert lens.tolist() == [250, 10]
    assert L.iq_cache_append(ctypes.byref(d), p, p, -1, p, None) == 1
    assert L.iq_cache_append(ctypes.byref(d), None, p, 1, p, None) == 1
    out = ctypes.c_size_t()
    assert L.iq_attend_workspace(ctypes.byref(d), 16, 1, ctypes.byref(out)) == 0 and out.value > 256
    # bad causal flag, rep not dividing 8, causal with too few tokens, missing workspace
    assert L.iq_attend(ctypes.byref(d), p, 16, 1, 0.0625, 2, p, p, 0, p, out.value, None) == 1
    assert L.iq_attend(ctypes.byref(d), p, 6, 1, 0.0625, 0, p, p, 0, p, out.value, None) == 4
    assert L.iq_attend(ctypes.byref(d), p, 16, 20, 0.0625, 1, p, p, 0, p, out.value, None) == 1
    assert L.iq_attend(ctypes.byref(d), p, 16, 1, 0.0625, 0, p, p, 0, None, 0, None) == 3
    assert L.iq_attend(ctypes.byref(d), p, 16, 1, 0.0625, 0, p, p, 0, p, 16, None) == 3
    d0, _ = fake_desc(lens=(0, 4))
    assert L.iq_attend(ctypes.byref(d0), p, 16, 1, 0.0625, 0, p, p, 0, p, out.value, None) == 1


def test_rotation_rejects(L):
    draws = np.zeros((64, 2, 4), dtype=np.float32)
    p = ctypes.c_void_p(0x20000000)
    assert L.iq_build_rotation(255, draws.ctypes.data, p, p, None) == 1
    assert L.iq_build_rotation(128, draws.ctypes.data, p, p, None) == 4
    assert L.iq_build_rotation(256, None, p, p, None) == 1


def test_debug_inject_and_noalloc_status_reject_bad_arguments(L):
    from rotated_bit_quantized_gb300._abi import IQ_INJECT_COMBINE_WAIT, IQ_INJECT_STAGE_NEVER_FILLED
    assert L.iq_debug_inject(4, 0, 0) == 1  # unknown flag
    assert b"flag" in L.iq_last_error()
    # a valid setting is host state only (it applies to this thread's next attention call), then clear it
    assert L.iq_debug_inject(IQ_INJECT_COMBINE_WAIT | IQ_INJECT_STAGE_NEVER_FILLED, 64, 1000000) == 0
    assert L.iq_debug_inject(0, 0, 0) == 0
    assert L.iq_noalloc_read_status(None, None) == 1  # null out pointer, checked before any device work


def test_cache_alloc_binds_and_validates(L):
    from rotated_bit_quantized_gb300._abi import IQCacheDesc
    d = IQCacheDesc()
    lens = np.array([7, 9], dtype=np.int32)
    P32 = ctypes.POINTER(ctypes.c_int32)
    bufs = (ctypes.c_void_p * 6)(*[0x10000000 + i * 0x1000000 for i in range(6)])
    assert L.iq_cache_alloc(ctypes.byref(d), 2, 2, 256, 64, 4, 3, 512, 0, bufs, lens.ctypes.data_as(P32)) == 0
    assert (d.batch, d.kv_heads, d.capacity, d.k_bits, d.v_bits, d.dtype) == (2, 2, 512, 4, 3, 0)
    assert d.v_biases == 0x15000000 and lens.tolist() == [0, 0]  # an empty cache
    assert L.iq_cache_alloc(ctypes.byref(d), 2, 2, 256, 64, 4, 3, 512, 1, bufs, lens.ctypes.data_as(P32)) == 0
    assert d.dtype == 1
    bad = (ctypes.c_void_p * 6)(*[0x10000008 + i * 0x1000000 for i in range(6)])  # not 16-byte aligned
    assert L.iq_cache_alloc(ctypes.byref(d), 2, 2, 256, 64, 4, 3, 512, 0, bad, lens.ctypes.data_as(P32)) == 1
    assert L.iq_cache_alloc(ctypes.byref(d), 2, 2, 256, 64, 7, 3, 512, 0, bufs, lens.ctypes.data_as(P32)) == 4
    assert L.iq_cache_alloc(ctypes.byref(d), 2, 2, 256, 64, 4, 3, 500, 0, bufs, lens.ctypes.data_as(P32)) == 1
    assert L.iq_cache_alloc(ctypes.byref(d), 2, 2, 256, 64, 4, 3, 512, 3, bufs, lens.ctypes.data_as(P32)) == 1


def test_cache_grow_rejects_before_copying(L):
    src, _ = fake_desc(batch=2, cap=256, lens=(100, 200))
    dst, dlens = fake_desc(batch=2, cap=512, lens=(0, 0))
    dst.k_codes = src.k_codes  # a shared buffer
    assert L.iq_cache_grow(ctypes.byref(src), ctypes.byref(dst), None) == 1
    small, _ = fake_desc(batch=2, cap=256, lens=(0, 0))
    for i, name in enumerate(("k_codes", "k_scales", "k_biases", "v_codes", "v_scales", "v_biases")):
        setattr(small, name, 0x40000000 + i * 0x1000000)
    big_src, _ = fake_desc(batch=2, cap=512, lens=(300, 10))
    assert L.iq_cache_grow(ctypes.byref(big_src), ctypes.byref(small), None) == 2  # dst capacity too small
    one, _ = fake_desc(batch=1, cap=512, lens=(0,))
    assert L.iq_cache_grow(ctypes.byref(src), ctypes.byref(one), None) == 1  # batch differs
    f32dst, _ = fake_desc(batch=2, cap=512, lens=(0, 0), dtype=1)
    for i, name in enumerate(("k_codes", "k_scales", "k_biases", "v_codes", "v_scales", "v_biases")):
        setattr(f32dst, name, 0x50000000 + i * 0x1000000)
    assert L.iq_cache_grow(ctypes.byref(src), ctypes.byref(f32dst), None) == 1  # dtype differs
