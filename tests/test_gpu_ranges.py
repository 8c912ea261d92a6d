"""Inputs at the edges of the fp16 operand ranges the attention kernels use.

The page computes in bf16 (`rotate_last` and `asym_quantized_sdpa` keep the
input dtype), whose range reaches ~3e38; the kernels feed fp16 operands to the
tensor cores.  They keep every case below inside fp16 exactly: queries enter as
q'' times a per-row power of two (rows with |q| up to 1e6, rows with entries
below 2^-14), and a large value scale raises the softmax reference so that
P * s_v stays below 2^15 (value groups spanning 1e4 and 1e6).  Each case runs
the decode kernel (1 query), the split-KV kernel with 32 rows per kv head
(4 queries) and, where it applies, the tensor-memory prefill kernel (16
queries x 8 heads = 128 rows per kv head), against the oracle.

Tolerance: the stated bar (max-abs 2e-3 with values ~N(0,1)) scaled by the
factor the values are multiplied by; attention is linear in the values, so the
same relative accuracy means that bar times the factor.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import attention
from oracle.cache import OracleCache
from parity_util import ATOL, compare_out, f32, oracle_blocks

pytestmark = pytest.mark.gpu

B, HKV, HQ, T = 2, 2, 16, 700


@pytest.fixture(scope="module")
def rot():
    from rotated_bit_quantized_gb300 import Rotation
    return Rotation(0, 256)


@pytest.fixture(scope="module")
def mb():
    return oracle_blocks(0)


def run_case(rot, mb, L, seed, qfun=None, vmul=1.0, causal=True):
    from rotated_bit_quantized_gb300 import IQCache
    k, v = si.kv_tokens(seed, B, HKV, T, outliers=True)
    v = (v.float() * vmul).bfloat16()
    q = si.queries(seed, B, HQ, L)
    if qfun is not None:
        q = qfun(q.float()).bfloat16()
    cache = IQCache(B, HKV)
    cache.reserve(T + 256)
    cache.append(k.cuda(), v.cuda(), rot)
    out = cache.attend(q.cuda(), rot, causal=causal, out_dtype=torch.float32)
    status = cache.device_status()
    oc = OracleCache(B, HKV)
    oc.append(f32(k), f32(v), mb)
    ref = attention.attend(f32(q), oc, mb, causal=causal)
    return out, ref, status


LS = [1, 4, 16]


@pytest.mark.parametrize("L", LS)
def test_queries_up_to_1e6(rot, mb, L):
    # max |q| ~ 1e6: q'' = bf16(q M_b) / 16 reaches ~1e5, past fp16's 65504
    out, ref, status = run_case(rot, mb, L, 31, qfun=lambda q: q * 3.0e5)
    assert status == 0
    assert float(np.abs(f32(si.queries(31, B, HQ, L)) * 3.0e5).max()) > 5e5
    compare_out(out, ref, f"|q| ~ 1e6, L={L}")


@pytest.mark.parametrize("L", LS)
def test_queries_with_entries_below_fp16_normal(rot, mb, L):
    # half the dims scaled by 1e-7: those q'' entries are ~1e-8, far below 2^-14
    def shrink(q):
        q = q.clone()
        q[..., 128:] *= 1e-7
        return q
    out, ref, status = run_case(rot, mb, L, 32, qfun=shrink)
    assert status == 0
    compare_out(out, ref, f"tiny q entries, L={L}")


@pytest.mark.parametrize("L", LS)
def test_tiny_queries(rot, mb, L):
    # every q'' ~ 1e-7: the softmax is nearly uniform
    out, ref, status = run_case(rot, mb, L, 33, qfun=lambda q: q * 1e-6)
    assert status == 0
    compare_out(out, ref, f"q ~ 1e-6, L={L}")


@pytest.mark.parametrize("L", LS)
def test_value_groups_spanning_1e4(rot, mb, L):
    # values x 2000: a 64-dim group spans ~1e4, value scales ~1.4e3 (> 2^9)
    out, ref, status = run_case(rot, mb, L, 34, vmul=2000.0)
    assert status == 0
    compare_out(out, ref, f"value range 1e4, L={L}", atol=ATOL * 2000.0)


@pytest.mark.parametrize("L", [1, 4])
def test_value_groups_spanning_1e6(rot, mb, L):
    # values x 2e5 on the split-KV kernels: value scales ~1.4e5, the reference moves by E = 9
    out, ref, status = run_case(rot, mb, L, 35, vmul=2.0e5)
    assert status == 0
    compare_out(out, ref, f"value range 1e6, L={L}", atol=ATOL * 2.0e5)


def test_prefill_refuses_values_beyond_fp16(rot, mb):
    # the tensor-memory prefill kernel takes dequantised values as fp16: a
    # value group spanning ~1e6 is reported (status bit 16), not silently wrong
    _, _, status = run_case(rot, mb, 16, 36, vmul=2.0e5)
    assert status & 16
