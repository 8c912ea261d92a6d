"""iq_cache_append_attend (append then attend in one call) on the GPU.

For decode-shaped steps it is a single attention launch whose CTAs encode the
new rows themselves, and for prefill-shaped steps (at least 128 query rows per
kv head) a single tensor-memory prefill launch whose CTAs claim and encode the
new rows' key tiles; the cache it leaves and the output it returns must equal
those of iq_cache_append followed by iq_attend bit for bit, and the output must
match the oracle within the attention bar.  Shapes that do not fuse (9 to 127
query rows per kv head, decode steps whose new rows cross a key tile) take the
two-launch path and must give the same results too.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import attention
from oracle.cache import OracleCache
from parity_util import compare_out, f32, oracle_blocks

pytestmark = pytest.mark.gpu

BUFS = ("k_codes", "k_scales", "k_biases", "v_codes", "v_scales", "v_biases")


@pytest.fixture(scope="module")
def rot():
    from rotated_bit_quantized_gb300 import Rotation
    return Rotation(0, 256)


@pytest.fixture(scope="module")
def mb():
    return oracle_blocks(0)


def _pair(rot, B, H, lens, seed):
    """Two identical device caches (ragged lengths) and the matching oracle cache."""
    from rotated_bit_quantized_gb300 import IQCache
    a, b = IQCache(B, H), IQCache(B, H)
    oc = OracleCache(B, H)
    T = max(lens)
    k, v = si.kv_tokens(seed, B, H, T, outliers=True)
    for c in (a, b):
        c.append(k.cuda(), v.cuda(), rot)
        c.trim(np.array([T - n for n in lens], dtype=np.int32))
    oc.append(f32(k), f32(v), oracle_blocks(0))
    oc.trim(np.array([T - n for n in lens]))
    return a, b, oc


def _same_cache(a, b):
    assert a.lens.tolist() == b.lens.tolist()
    for name in BUFS:
        x, y = getattr(a, name), getattr(b, name)
        for s in range(a.batch):
            n = int(a.lens[s])
            assert torch.equal(x[s, :, :n], y[s, :, :n]), f"{name} sequence {s} differs"


@pytest.mark.parametrize("lens,n,Hq,L,causal", [
    ([300, 511, 256], 1, 16, 1, True),    # fused: decode, ragged (511 -> last row of a tile, 256 -> first)
    ([1000, 37], 1, 16, 1, False),        # fused, no mask
    ([200, 130], 3, 2, 4, True),          # fused: 1 head per kv head x 4 queries = 4 rows
    ([126, 300], 4, 16, 4, True),         # two launches: 32 query rows per kv head, rows 126..129 cross a tile
    ([300, 77], 200, 16, 200, True),      # fused prefill: 1600 rows per kv head, new rows start inside a key tile
    ([64, 130], 150, 8, 150, False),      # fused prefill, no mask: 600 rows per kv head
])
def test_append_attend_equals_two_calls(rot, mb, lens, n, Hq, L, causal):
    B, H = len(lens), 2
    a, b, oc = _pair(rot, B, H, lens, seed=71)
    k, v = si.kv_tokens(72, B, H, n, outliers=True, step=1)
    q = si.queries(73, B, Hq, L)
    out_a = a.append_attend(k.cuda(), v.cuda(), q.cuda(), rot, causal=causal, out_dtype=torch.float32)
    b.append(k.cuda(), v.cuda(), rot)
    out_b = b.attend(q.cuda(), rot, causal=causal, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert a.device_status() == 0 and b.device_status() == 0
    _same_cache(a, b)
    assert torch.equal(out_a, out_b)
    oc.append(f32(k), f32(v), mb)
    ref = attention.attend(f32(q), oc, mb, causal=causal)
    compare_out(out_a, ref, f"append_attend lens={lens} n={n} Hq={Hq} L={L}")


def test_decode_loop_with_trims(rot, mb):
    """Several fused steps in a row with a trim in between, bf16 output, against the oracle."""
    B, H = 2, 2
    a, _, oc = _pair(rot, B, H, [255, 640], seed=81)
    for step in range(4):
        k, v = si.kv_tokens(82, B, H, 1, outliers=True, step=step)
        q = si.queries(83, B, 16, 1, step=step)
        out = a.append_attend(k.cuda(), v.cuda(), q.cuda(), rot, causal=True)
        torch.cuda.synchronize()
        oc.append(f32(k), f32(v), mb)
        compare_out(out, attention.attend(f32(q), oc, mb, causal=True), f"step {step}")
        if step == 1:
            a.trim(np.array([1, 0], dtype=np.int32))
            oc.trim(np.array([1, 0]))
    assert a.device_status() == 0


def test_prefill_chunks_fused(rot, mb):
    """Chunked prefill through the fused call (chunks of 192 new rows, a trim
    between chunks): each chunk's cache equals the two-call path's, each output
    matches the oracle."""
    B, H, Hq, n = 1, 2, 16, 192
    a, b, oc = _pair(rot, B, H, [40], seed=91)
    for step in range(3):
        k, v = si.kv_tokens(92, B, H, n, outliers=True, step=step)
        q = si.queries(93, B, Hq, n, step=step)
        out_a = a.append_attend(k.cuda(), v.cuda(), q.cuda(), rot, causal=True, out_dtype=torch.float32)
        b.append(k.cuda(), v.cuda(), rot)
        out_b = b.attend(q.cuda(), rot, causal=True, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert a.device_status() == 0 and b.device_status() == 0
        _same_cache(a, b)
        assert torch.equal(out_a, out_b)
        oc.append(f32(k), f32(v), mb)
        compare_out(out_a, attention.attend(f32(q), oc, mb, causal=True), f"chunk {step}")
        if step == 0:
            for c in (a, b):
                c.trim(np.array([100], dtype=np.int32))
            oc.trim(np.array([100]))


def test_prefill_append_is_one_kernel(rot):
    """A prefill-shaped append_attend launches the prefill kernel alone (its
    CTAs encode the new rows); the separate append kernel does not run."""
    from torch.profiler import ProfilerActivity, profile
    B, H, Hq, n = 1, 2, 16, 256
    a, _, _ = _pair(rot, B, H, [500], seed=95)
    k, v = si.kv_tokens(96, B, H, n, outliers=True)
    q = si.queries(97, B, Hq, n)
    kd, vd, qd = k.cuda(), v.cuda(), q.cuda()
    a.append_attend(kd, vd, qd, rot, causal=True)  # warm-up (workspace, attributes)
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        a.append_attend(kd, vd, qd, rot, causal=True)
        torch.cuda.synchronize()
    kernels = [e.key for e in prof.key_averages() if "kernel" in e.key]
    if not kernels:
        pytest.skip("the profiler recorded no GPU kernels on this machine")
    assert any("prefill_kernel" in x for x in kernels), kernels
    assert not any("append_kernel" in x for x in kernels), kernels
    assert a.device_status() == 0


def test_prefill_status_clean_over_many_calls(rot):
    """Many prefill launches back to back (fused and two-call, 512-row chunks)
    end with a clean status word: no bounded wait of the tensor-memory kernel's
    pipeline ever runs out (a barrier phase two ahead of its waiter would look
    incomplete and stall until the limit)."""
    from rotated_bit_quantized_gb300 import IQCache
    B, H, Hq, n = 1, 2, 16, 512
    a, b = IQCache(B, H), IQCache(B, H)
    for c in (a, b):
        c.reserve(24 * n + 256)
    for step in range(24):
        k, v = si.kv_tokens(98, B, H, n, outliers=True, step=step)
        q = si.queries(99, B, Hq, n, step=step)
        kd, vd, qd = k.cuda(), v.cuda(), q.cuda()
        a.append_attend(kd, vd, qd, rot, causal=True)
        b.append(kd, vd, rot)
        b.attend(qd, rot, causal=True)
    torch.cuda.synchronize()
    assert a.device_status() == 0 and b.device_status() == 0
