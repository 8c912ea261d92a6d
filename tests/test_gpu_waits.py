"""Bounded device waits run out on purpose, through the library's injection
hook (iq_debug_inject: host-side settings for the next call; no kernel faults,
traps or waits without a limit).  Each case checks that the failing call
returns, that its status word says which wait ran out, and that the next call
on the same workspace is correct (the combine's unit counters return to zero
also after a timeout)."""
import ctypes

import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import attention
from oracle.cache import OracleCache
from parity_util import compare_out, f32, oracle_blocks

pytestmark = pytest.mark.gpu

B, HKV, HQ, T = 4, 2, 16, 3000  # 8 units of 24 tiles over ~24 tile ranges: every unit is shared (combine)


@pytest.fixture(scope="module")
def setup():
    from rotated_bit_quantized_gb300 import IQCache, Rotation
    rot = Rotation(0, 256)
    k, v = si.kv_tokens(71, B, HKV, T, outliers=True)
    cache = IQCache(B, HKV)
    cache.reserve(T + 256)
    cache.append(k.cuda(), v.cuda(), rot)
    oc = OracleCache(B, HKV)
    oc.append(f32(k), f32(v), oracle_blocks(0))
    return rot, cache, oc


def _inject(flags, spin_limit=0, wait_ns=0):
    from rotated_bit_quantized_gb300._abi import lib
    assert lib().iq_debug_inject(flags, spin_limit, wait_ns) == 0


@pytest.mark.parametrize("flags,spin,wait_ns,bit", [(1, 0, 1_000_000, 8), (2, 64, 0, 2)])
def test_wait_runs_out_then_next_call_is_correct(setup, flags, spin, wait_ns, bit):
    rot, cache, oc = setup
    mb = oracle_blocks(0)
    assert cache.device_status() == 0
    q = si.queries(72, B, HQ, 1).cuda()
    _inject(flags, spin, wait_ns)
    cache.attend(q, rot, causal=False, out_dtype=torch.float32)  # returns; its output is not meaningful
    st = cache.device_status()  # synchronises and clears
    assert st & bit, f"status {st:#x} lacks bit {bit}"
    for call in range(2):  # the calls after it are correct, with a clean status
        q = si.queries(73 + call, B, HQ, 1)
        out = cache.attend(q.cuda(), rot, causal=False, out_dtype=torch.float32)
        compare_out(out, attention.attend(f32(q), oc, mb), f"after injected failure {flags}, call {call}")
        assert cache.device_status() == 0


def test_fused_prefill_row_wait_runs_out_then_next_call_is_correct():
    """The fused prefill's wait for its new rows, made to run out from the host:
    the workspace's chunk counter is preset past every chunk (2^30 takes), so
    no CTA encodes and every producer's row count stays below n.  The call
    returns within the waits' limits with status bit 0x20000; the grid leaves
    its counters at zero, so the same call after a trim is correct."""
    from rotated_bit_quantized_gb300 import IQCache, Rotation
    rot = Rotation(0, 256)
    mb = oracle_blocks(0)
    B, H, Hq, n = 1, 2, 16, 256  # 2048 query rows per kv head: 32 CTAs, one wave
    cache = IQCache(B, H)
    k0, v0 = si.kv_tokens(74, B, H, 300, outliers=True)
    cache.append(k0.cuda(), v0.cuda(), rot)
    oc = OracleCache(B, H)
    oc.append(f32(k0), f32(v0), mb)
    k, v = si.kv_tokens(75, B, H, n, outliers=True, step=1)
    q = si.queries(76, B, Hq, n)
    cache.append_attend(k.cuda(), v.cuda(), q.cuda(), rot, causal=True)  # creates the workspace
    cache.trim(n)
    assert cache.device_status() == 0
    cache._workspace[256:260].view(torch.int32)[0] = 1 << 30  # the unit-counter area: chunks taken
    cache.append_attend(k.cuda(), v.cuda(), q.cuda(), rot, causal=True)  # returns; its output is not meaningful
    torch.cuda.synchronize()
    # the grid's last CTA zeroed the counters (taken, finished, rows per kv head)
    # before the status read below, which would also clear them after a failure
    assert cache._workspace[256:256 + 4 * (2 + B * H)].view(torch.int32).tolist() == [0] * (2 + B * H)
    st = cache.device_status()
    assert st & 0x20000, f"status {st:#x} lacks the fused append's wait bit"
    cache.trim(n)
    out = cache.append_attend(k.cuda(), v.cuda(), q.cuda(), rot, causal=True, out_dtype=torch.float32)
    assert cache.device_status() == 0
    oc.append(f32(k), f32(v), mb)
    compare_out(out, attention.attend(f32(q), oc, mb, causal=True), "fused prefill after an injected wait failure")
