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
    """Every chunk: its first and last 64 queries and 256 seeded random ones,
    all 16 heads, against the oracle; every stored row bit-exact."""
    from rotated_bit_quantized_gb300 import IQCache
    w = si.WORKLOADS[3]
    cache = IQCache(1, 2)
    cache.reserve(16 * 2048)
    oc = OracleCache(1, 2)
    rng = np.random.default_rng(333)
    for c in range(16):
        k, v = si.kv_tokens(w["seed"], 1, 2, 2048, outliers=True, step=c)
        q = si.queries(w["seed"], 1, 16, 2048, step=c)
        out = cache.append_attend(k.cuda(), v.cuda(), q.cuda(), rot, causal=True, out_dtype=torch.float32)
        oc.append(f32(k), f32(v), mb)
        qi = np.unique(np.concatenate([np.arange(64), np.arange(2048 - 64, 2048), rng.integers(0, 2048, 256)]))
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


def test_workload4_batched_decode_as_benchmarked(rot, mb):
    """The benchmarked call at full size, as bench.py issues it: three warm-up
    steps, a trim back to the 32768-token prefill, then 8 consecutive
    append + attend calls back to back with no synchronisation in between (each
    call's attention grid streams while the previous call's grids finish, and
    the first one after the trim waits before its fused encode).  Every step is
    checked against the oracle on three sequences, and the new rows bit-exact."""
    w = si.WORKLOADS[4]
    W, K = 3, 8
    cache = device_prefill(w, rot)
    base = cache.lens.copy()
    steps = []
    for s in range(W + K):
        k, v = si.kv_tokens(w["seed"], 32, 2, 1, outliers=True, step=s)
        q = si.queries(w["seed"], 32, 16, 1, step=s)
        steps.append((k.cuda(), v.cuda(), q.cuda()))
    scratch = torch.empty((32, 16, 1, 256), dtype=torch.bfloat16, device="cuda")
    for s in range(W):
        cache.append_attend(*steps[s], rot, causal=True, out=scratch)
    cache.trim(cache.lens - base)
    outs = [torch.empty((32, 16, 1, 256), dtype=torch.bfloat16, device="cuda") for _ in range(K)]
    for i in range(K):
        cache.append_attend(*steps[W + i], rot, causal=True, out=outs[i])
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    for b in (0, 17, 31):
        oc = oracle_sequence(w, b, mb)
        for i in range(K):
            new = [si.kv_slice(w["seed"], b, h, 1, outliers=True, step=W + i) for h in range(2)]
            oc.append(np.stack([f32(x[0]) for x in new])[None], np.stack([f32(x[1]) for x in new])[None], mb)
            q = si.queries(w["seed"], 32, 16, 1, step=W + i)[b:b + 1]
            ref = np.full(outs[i].shape, np.nan)
            ref[b] = attention.attend(f32(q), oc, mb, causal=True)[0]
            compare_out(outs[i], ref, f"workload 4 step {i} seq {b}")
        n = 32768 + K
        for h in range(2):
            for name, want in (("k_codes", oc.k[0]), ("v_codes", oc.v[0])):
                got = getattr(cache, name)[b, h, 32768:n].cpu().numpy().view(np.uint32)
                assert np.array_equal(got, want[0, h, 32768:n]), f"{name} new rows of seq {b}"
            for name, want in (("k_scales", oc.k[1]), ("k_biases", oc.k[2]), ("v_scales", oc.v[1]),
                               ("v_biases", oc.v[2])):
                got = getattr(cache, name)[b, h, 32768:n].float().cpu().numpy()
                np.testing.assert_array_equal(got, want[0, h, 32768:n])


def test_workload5_speculative_verify(rot, mb):
    """All 32 verify steps (append 4 drafts, attend 4 causal queries, trim the
    rejected suffix) on the full 8 x 131072-token caches; steps 0, 1, 15 and
    31 checked in full (every sequence, head and query) against the oracle."""
    w = si.WORKLOADS[5]
    B, steps = 8, w["steps"]
    cache = device_prefill(w, rot)
    acc = si.accepted_lengths(steps, B, 4, w["accept_seed"])
    checked = (0, 1, 15, 31)
    outs, qs = {}, {}
    for s in range(steps):
        k, v = si.kv_tokens(w["seed"], B, 2, 4, outliers=True, step=s)
        q = si.queries(w["seed"], B, 16, 4, step=s)
        out = cache.append_attend(k.cuda(), v.cuda(), q.cuda(), rot, causal=True, out_dtype=torch.float32)
        if s in checked:
            outs[s], qs[s] = out, q
        cache.commit_verified_prefix(4, acc[s])
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    for b in range(B):
        oc = oracle_sequence(w, b, mb)
        for s in range(steps):
            new = [si.kv_slice(w["seed"], b, h, 4, outliers=True, step=s) for h in range(2)]
            oc.append(np.stack([f32(x[0]) for x in new])[None], np.stack([f32(x[1]) for x in new])[None], mb)
            if s in checked:
                ref = np.full(outs[s].shape, np.nan)
                ref[b] = attention.attend(f32(qs[s][b:b + 1]), oc, mb, causal=True)[0]
                compare_out(outs[s], ref, f"workload 5 step {s} seq {b}")
            oc.trim(4 - int(acc[s, b]))
        assert int(oc.lens[0]) == int(cache.lens[b])
