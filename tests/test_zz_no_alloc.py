"""iq_attend_noalloc, the attention entry point for callers that cannot
allocate device memory (their allocator owns all of HBM, they only see the
buffers a host hands them, or an allocation would stall a latency-bound
decode loop).  It must give the same result as iq_attend with a caller
workspace, on two calls in a row (the shared scratch keeps the previous call's
contents), and reject calls whose scratch need exceeds its fixed size.

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
    return lib().iq_attend_noalloc(ctypes.byref(d), ctypes.c_void_p(q.data_ptr()), q.shape[1], q.shape[2],
                                   1.0 / 16, 1 if causal else 0, ctypes.c_void_p(rot.blocks_bf16.data_ptr()),
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


def test_noalloc_rejects_calls_above_its_scratch():
    from rotated_bit_quantized_gb300 import IQCache, Rotation
    from rotated_bit_quantized_gb300._abi import IQ_ERR_WORKSPACE, IQ_NOALLOC_SCRATCH_BYTES, lib
    rot = Rotation(0, 256)
    cache = IQCache(1, 2)
    k, v = si.kv_tokens(63, 1, 2, 8192, outliers=True)
    cache.append(k.cuda(), v.cuda(), rot)
    L = 8192  # a long causal query block needs far more partials than the scratch holds
    assert cache.workspace_bytes(16, L) > IQ_NOALLOC_SCRATCH_BYTES
    q = si.queries(64, 1, 16, L).cuda()
    out = torch.empty((1, 16, L, 256), dtype=torch.float32, device="cuda")
    assert _call_noalloc(cache, q, rot, True, out) == IQ_ERR_WORKSPACE
    assert b"scratch" in lib().iq_last_error()
