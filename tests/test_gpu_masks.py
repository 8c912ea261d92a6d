"""Explicit attention masks (iq_attend_mask) against the oracle on the GPU.

The page's `asym_quantized_sdpa` takes a bool mask (masked scores replaced by
the dtype's most negative value) or a float mask (added to the scores).  Masks
are [B, L, S] (S >= every length), shared by the heads.  Bars as the other
attention tests (max-abs 2e-3 on the fp32 output); special cases: the causal
pattern as a mask equals the causal path, an all-kept mask equals no mask, and
a row whose keys are all masked by a bool mask is the uniform mean.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import attention
from parity_util import compare_out, f32, oracle_blocks

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rot():
    from rotated_bit_quantized_gb300 import Rotation
    return Rotation(0, 256)


@pytest.fixture(scope="module")
def mb():
    return oracle_blocks(0)


def _caches(rot, mb, lens, seed):
    from oracle.cache import OracleCache
    from rotated_bit_quantized_gb300 import IQCache
    B, H = len(lens), 2
    T = max(lens)
    k, v = si.kv_tokens(seed, B, H, T, outliers=True)
    cache = IQCache(B, H)
    cache.append(k.cuda(), v.cuda(), rot)
    oc = OracleCache(B, H)
    oc.append(f32(k), f32(v), mb)
    cut = np.array([T - n for n in lens], dtype=np.int32)
    cache.trim(cut)
    oc.trim(cut)
    return cache, oc


def _masks(seed, B, L, S, lens):
    rng = np.random.default_rng(seed)
    keep = rng.random((B, L, S)) < 0.7
    add = rng.standard_normal((B, L, S)).astype(np.float32) * 2
    add[rng.random((B, L, S)) < 0.2] = -np.inf
    for b, n in enumerate(lens):  # every float-mask row keeps at least one key
        add[b, :, n - 1] = 0.0
    return keep, add


@pytest.mark.parametrize("lens,Hq,L", [([700, 129], 16, 1), ([300, 1025, 64], 16, 4), ([5000], 2, 3)])
def test_masks_match_oracle(rot, mb, lens, Hq, L):
    cache, oc = _caches(rot, mb, lens, seed=91)
    B, S = len(lens), max(lens) + 3
    q = si.queries(92, B, Hq, L)
    keep, add = _masks(93, B, L, S, lens)
    keep[0, L - 1, :] = False  # a row with every key masked
    for m in (keep, add):
        got = cache.attend(q.cuda(), rot, mask=torch.from_numpy(m).cuda(), out_dtype=torch.float32)
        torch.cuda.synchronize()
        ref = attention.attend(f32(q), oc, mb, mask=m)
        compare_out(got, ref, f"mask {m.dtype} lens={lens} Hq={Hq} L={L}")
    assert cache.device_status() == 0


def test_mask_special_cases_on_gpu(rot, mb):
    lens = [333, 2049]
    cache, oc = _caches(rot, mb, lens, seed=95)
    B, L, S = 2, 4, 2052
    q = si.queries(96, B, 16, L).cuda()
    causal = cache.attend(q, rot, causal=True, out_dtype=torch.float32)
    plain = cache.attend(q, rot, out_dtype=torch.float32)
    pos = np.array(lens)[:, None] - L + np.arange(L)[None, :]
    keep = np.arange(S)[None, None, :] <= pos[:, :, None]
    as_keep = cache.attend(q, rot, mask=torch.from_numpy(keep).cuda(), out_dtype=torch.float32)
    as_add = cache.attend(q, rot, mask=torch.from_numpy(np.where(keep, 0.0, -np.inf).astype(np.float32)).cuda(),
                          out_dtype=torch.float32)
    all_kept = cache.attend(q, rot, mask=torch.ones((B, L, S), dtype=torch.bool, device="cuda"),
                            out_dtype=torch.float32)
    torch.cuda.synchronize()
    for got in (as_keep, as_add):
        np.testing.assert_allclose(got.cpu().numpy(), causal.cpu().numpy(), atol=2e-3)
    np.testing.assert_allclose(all_kept.cpu().numpy(), plain.cpu().numpy(), atol=2e-3)
    with pytest.raises(ValueError):
        cache.attend(q, rot, causal=True, mask=torch.from_numpy(keep).cuda())
    assert cache.device_status() == 0
