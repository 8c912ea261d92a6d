"""iq_attend_noalloc, the attention entry point for callers that cannot
allocate device memory (their allocator owns all of HBM, they only see the
buffers a host hands them, or an allocation would stall a latency-bound
decode loop).  It must give the same result as iq_attend with a caller
workspace, on two calls in a row (the shared scratch keeps the previous call's
contents), on the split-KV, generic-format, two-launch and prefill paths;
report kernel failures through iq_noalloc_read_status; keep its counters
consistent after a wait that ran out; and reject calls whose scratch need
exceeds its fixed size.

This file is collected last so that a failure here cannot hide another test.
"""
import ctypes

import numpy as np
import pytest
import torch

import seeded_inputs as si
from parity_util import ATOL

pytestmark = pytest.mark.gpu


def _call_noalloc(cache, q, rot, causal, out):
    from rotated_bit_quantized_gb300._abi import lib
    d = cache.desc()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    blocks = rot.blocks_f32 if cache.dtype == torch.float32 else rot.blocks_bf16
    return lib().iq_attend_noalloc(ctypes.byref(d), ctypes.c_void_p(q.data_ptr()), q.shape[1], q.shape[2],
                                   1.0 / 16, 1 if causal else 0, ctypes.c_void_p(blocks.data_ptr()),
                                   ctypes.c_void_p(out.data_ptr()), 1 if out.dtype == torch.float32 else 0,
                                   stream)


@pytest.mark.parametrize("B,T,L,causal", [(4, 3000, 1, True), (2, 777, 4, True), (1, 256, 1, False)])
def test_noalloc_matches_workspace_path_twice(B, T, L, causal):
    from rotated_bit_quantized_gb300 import IQCache, Rotation
    rot = Rotation(0, 256)
    cache = IQCache(B, 2)
    k, v = si.kv_tokens(61, B, 2, T, outliers=True)
    cache.append(k.cuda(), v.cuda(), rot)
    for call in range(2):
        q = si.queries(62 + call, B, 16, L).cuda()
        ref = cache.attend(q, rot, causal=causal, out_dtype=torch.float32)
        out = torch.full_like(ref, float("nan"))
        assert _call_noalloc(cache, q, rot, causal, out) == 0
        torch.cuda.synchronize()
        err = (out - ref).abs().max().item()
        assert err <= ATOL, f"call {call}: max abs difference {err}"
        assert torch.isfinite(out).all()
        outb = torch.empty(ref.shape, dtype=torch.bfloat16, device=ref.device)
        assert _call_noalloc(cache, q, rot, causal, outb) == 0
        refb = cache.attend(q, rot, causal=causal, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert (outb.float() - refb.float()).abs().max().item() <= ATOL + 2 ** -7
    assert cache.device_status() == 0


def _read_noalloc_status():
    from rotated_bit_quantized_gb300._abi import lib
    st = ctypes.c_int(-1)
    code = lib().iq_noalloc_read_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), ctypes.byref(st))
    return code, st.value


def _ref_and_noalloc(cache, rot, q, causal):
    ref = cache.attend(q, rot, causal=causal, out_dtype=torch.float32)
    out = torch.full_like(ref, float("nan"))
    assert _call_noalloc(cache, q, rot, causal, out) == 0
    torch.cuda.synchronize()
    return ref, out


@pytest.mark.parametrize("fmt,B,H,Hq,T,L", [
    ((2, 8, 128), 2, 2, 16, 900, 1),   # a generic format (K2 / V8, groups of 128)
    ((4, 3, 64), 256, 8, 64, 256, 1),  # 2048 query tiles: two launches share the scratch
    ((4, 3, 64), 1, 2, 16, 700, 16),   # 128 rows per kv head: the tensor-memory prefill kernel
])
def test_noalloc_other_paths(fmt, B, H, Hq, T, L):
    from rotated_bit_quantized_gb300 import IQCache, Rotation
    rot = Rotation(0, 256)
    cache = IQCache(B, H, k_bits=fmt[0], v_bits=fmt[1], group_size=fmt[2])
    k, v = si.kv_tokens(65, B, H, T, outliers=True)
    cache.append(k.cuda(), v.cuda(), rot)
    for call in range(2):
        q = si.queries(66 + call, B, Hq, L).cuda()
        ref, out = _ref_and_noalloc(cache, rot, q, True)
        err = (out - ref).abs().max().item()
        assert err <= ATOL, f"call {call}: max abs difference {err}"
    assert _read_noalloc_status() == (0, 0)
    assert cache.device_status() == 0


def test_noalloc_float32_cache():
    """A float32 cache (float32 queries, scales and biases; the generic path)
    through the no-allocation entry point: the same result as with a caller
    workspace."""
    from rotated_bit_quantized_gb300 import IQCache, Rotation
    rot = Rotation(0, 256)
    cache = IQCache(2, 2, dtype=torch.float32)
    k, v = si.kv_tokens(64, 2, 2, 1200, outliers=True, dtype=torch.float32)
    cache.append(k.cuda(), v.cuda(), rot)
    for call in range(2):
        q = si.queries(70 + call, 2, 16, 2, dtype=torch.float32).cuda()
        ref, out = _ref_and_noalloc(cache, rot, q, True)
        assert (out - ref).abs().max().item() <= 1e-6
    assert _read_noalloc_status() == (0, 0)
    assert cache.device_status() == 0


def test_noalloc_status_and_counters_after_a_wait_runs_out():
    """A combine wait that runs out (injected) is reported by
    iq_noalloc_read_status; the unit counters of the shared scratch are back at
    zero without any clearing, so the next call is correct before the status
    is even read."""
    from rotated_bit_quantized_gb300 import IQCache, Rotation
    from rotated_bit_quantized_gb300._abi import IQ_ERR_DEVICE, IQ_INJECT_COMBINE_WAIT, lib
    rot = Rotation(0, 256)
    cache = IQCache(4, 2)
    k, v = si.kv_tokens(67, 4, 2, 3000, outliers=True)
    cache.append(k.cuda(), v.cuda(), rot)
    assert _read_noalloc_status() == (0, 0)
    q = si.queries(68, 4, 16, 1).cuda()
    out = torch.empty((4, 16, 1, 256), dtype=torch.float32, device="cuda")
    assert lib().iq_debug_inject(IQ_INJECT_COMBINE_WAIT, 0, 1_000_000) == 0
    assert _call_noalloc(cache, q, rot, False, out) == 0
    q2 = si.queries(69, 4, 16, 1).cuda()
    ref, out2 = _ref_and_noalloc(cache, rot, q2, False)  # no status read in between
    assert (out2 - ref).abs().max().item() <= ATOL
    code, st = _read_noalloc_status()
    assert code == IQ_ERR_DEVICE and st & 8
    assert _read_noalloc_status() == (0, 0)  # cleared
    ref, out3 = _ref_and_noalloc(cache, rot, q, False)
    assert (out3 - ref).abs().max().item() <= ATOL
    assert _read_noalloc_status() == (0, 0)


def test_noalloc_rejects_calls_above_its_scratch():
    from rotated_bit_quantized_gb300 import IQCache, Rotation
    from rotated_bit_quantized_gb300._abi import IQ_ERR_WORKSPACE, IQ_NOALLOC_SCRATCH_BYTES, lib
    rot = Rotation(0, 256)
    # 64 sequences x 2 kv heads x 8 query tiles of 16 rows (15 queries x 8
    # heads = 120 rows per kv head: the split-KV kernel): 1024 units, whose
    # partials need more than the scratch holds
    B, L = 64, 15
    cache = IQCache(B, 2)
    k, v = si.kv_tokens(63, B, 2, 256, outliers=True)
    cache.append(k.cuda(), v.cuda(), rot)
    assert cache.workspace_bytes(16, L) > IQ_NOALLOC_SCRATCH_BYTES
    q = si.queries(64, B, 16, L).cuda()
    out = torch.empty((B, 16, L, 256), dtype=torch.float32, device="cuda")
    assert _call_noalloc(cache, q, rot, True, out) == IQ_ERR_WORKSPACE
    assert b"scratch" in lib().iq_last_error()
