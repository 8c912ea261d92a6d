"""The five workloads at their full sizes, in the benchmark's launch
configuration, checked against the oracle on sampled sequences / queries (the
oracle rebuilds only the slices it samples from the seeded generators)."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import attention
from oracle.cache import OracleCache
from parity_util import assert_rows_equal, compare_out, f32, oracle_blocks

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rot():
    from rotated_bit_quantized_gb300 import Rotation
    return Rotation(0, 256)


@pytest.fixture(scope="module")
def mb():
    return oracle_blocks(0)


def device_prefill(w, rot):
    from rotated_bit_quantized_gb300 import IQCache
    cache = IQCache(w["B"], w["Hkv"])
    cache.reserve(w["prefill"] + max(1, w["steps"]) * w["append"] + 256)
    if w["prefill"]:
        k, v = si.kv_tokens(w["seed"], w["B"], w["Hkv"], w["prefill"], outliers=w["outliers"])
        for lo in range(0, w["prefill"], 8192):
            hi = min(lo + 8192, w["prefill"])
            cache.append(k[:, :, lo:hi].cuda(), v[:, :, lo:hi].cuda(), rot)
    return cache


def oracle_sequence(w, b, mb, steps=0, trims=None):
    """Oracle cache of sequence b alone: prefill, then `steps` appends with per-step trims."""
    oc = OracleCache(1, w["Hkv"])

    def add(n, step):
        pairs = [si.kv_slice(w["seed"], b, h, n, outliers=w["outliers"], step=step) for h in range(w["Hkv"])]
        oc.append(np.stack([f32(p[0]) for p in pairs])[None], np.stack([f32(p[1]) for p in pairs])[None], mb)

    if w["prefill"]:
        add(w["prefill"], None)
    for s in range(steps):
        add(w["append"], s)
        if trims is not None and s < steps - 1:
            oc.trim(trims[s])
    return oc


def test_workload1_tiny(rot, mb):
    w = si.WORKLOADS[1]
    cache = device_prefill(w, rot)
    q = si.queries(w["seed"], 1, 1, 1)
    out = cache.attend(q.cuda(), rot, out_dtype=torch.float32)
    oc = oracle_sequence(w, 0, mb)
    compare_out(out, attention.attend(f32(q), oc, mb), "workload 1")
    kk, vv = si.kv_tokens(w["seed"], 1, 1, 256)
    assert_rows_equal(cache, 0, 0, 0, 256, f32(kk[0, 0]), f32(vv[0, 0]), mb)


def test_workload2_single_stream_decode(rot, mb):
    w = si.WORKLOADS[2]
    cache = device_prefill(w, rot)
    q = si.queries(w["seed"], 1, 16, 1)
    oc = oracle_sequence(w, 0, mb)
    ref = attention.attend(f32(q), oc, mb)
    for dt in (torch.float32, torch.bfloat16):
        compare_out(cache.attend(q.cuda(), rot, out_dtype=dt), ref, f"workload 2 {dt}")
    for h in range(2):
        kk, vv = si.kv_slice(w["seed"], 0, h, 4096, outliers=True)
        assert_rows_equal(cache, 0, h, 0, 4096, f32(kk), f32(vv), mb)


def test_workload3_chunked_prefill(rot, mb):
    from rotated_bit_quantized_gb300 import IQCache
    w = si.WORKLOADS[3]
    cache = IQCache(1, 2)
    cache.reserve(16 * 2048)
    oc = OracleCache(1, 2)
    rng = np.random.default_rng(333)
    checked = {0, 5, 15}
    for c in range(16):
        k, v = si.kv_tokens(w["seed"], 1, 2, 2048, outliers=True, step=c)
        cache.append(k.cuda(), v.cuda(), rot)
        oc.append(f32(k), f32(v), mb)
        q = si.queries(w["seed"], 1, 16, 2048, step=c)
        out = cache.attend(q.cuda(), rot, causal=True, out_dtype=torch.float32)
        if c in checked:
            qi = np.unique(np.concatenate([np.arange(8), np.arange(2040, 2048), rng.integers(0, 2048, 16)]))
            ref = attention.attend(f32(q), oc, mb, causal=True, query_index=qi)
            compare_out(out, ref, f"workload 3 chunk {c}")
    assert cache.device_status() == 0
    for h in range(2):
        got = cache.k_codes[0, h, :32768].cpu().numpy().view(np.uint32)
        assert np.array_equal(got, oc.k[0][0, h, :32768])
        got = cache.v_codes[0, h, :32768].cpu().numpy().view(np.uint32)
        assert np.array_equal(got, oc.v[0][0, h, :32768])
    cache.trim(w["trim_after"])
    oc.trim(w["trim_after"])
    assert cache.lens.tolist() == [31768]
    q = si.queries(w["seed"], 1, 16, 1, step=99)
    compare_out(cache.attend(q.cuda(), rot, out_dtype=torch.float32), attention.attend(f32(q), oc, mb),
                "workload 3 after trim")


def test_workload4_batched_decode(rot, mb):
    w = si.WORKLOADS[4]
    cache = device_prefill(w, rot)
    sampled = (0, 17, 31)
    for s in range(2):
        k, v = si.kv_tokens(w["seed"], 32, 2, 1, outliers=True, step=s)
        q = si.queries(w["seed"], 32, 16, 1, step=s)
        cache.append(k.cuda(), v.cuda(), rot)
        out = cache.attend(q.cuda(), rot, causal=True, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        for b in sampled if s == 1 else (0,):
            oc = oracle_sequence(w, b, mb, steps=s + 1)
            ref = np.full(out.shape, np.nan)
            ref[b] = attention.attend(f32(q[b:b + 1]), oc, mb, causal=True)[0]
            compare_out(out, ref, f"workload 4 step {s} seq {b}")
            if s == 1 and b == 17:
                for h in range(2):
                    got = cache.k_codes[b, h, :32770].cpu().numpy().view(np.uint32)
                    assert np.array_equal(got, oc.k[0][0, h, :32770])
                    got = cache.v_codes[b, h, :32770].cpu().numpy().view(np.uint32)
                    assert np.array_equal(got, oc.v[0][0, h, :32770])
    assert cache.device_status() == 0


def test_workload5_speculative_verify(rot, mb):
    w = si.WORKLOADS[5]
    cache = device_prefill(w, rot)
    acc = si.accepted_lengths(w["steps"], 8, 4, w["accept_seed"])
    sampled = (0, 6)
    steps = 3
    for s in range(steps):
        k, v = si.kv_tokens(w["seed"], 8, 2, 4, outliers=True, step=s)
        q = si.queries(w["seed"], 8, 16, 4, step=s)
        cache.append(k.cuda(), v.cuda(), rot)
        out = cache.attend(q.cuda(), rot, causal=True, out_dtype=torch.float32)
        torch.cuda.synchronize()
        if s == steps - 1:
            rejected = [4 - acc[t] for t in range(steps)]
            for b in sampled:
                oc = oracle_sequence(w, b, mb, steps=s + 1, trims=[r[b] for r in rejected])
                assert int(oc.lens[0]) == int(cache.lens[b])
                ref = np.full(out.shape, np.nan)
                ref[b] = attention.attend(f32(q[b:b + 1]), oc, mb, causal=True)[0]
                compare_out(out, ref, f"workload 5 step {s} seq {b}")
        cache.commit_verified_prefix(4, acc[s])
    assert cache.device_status() == 0
