"""The page's snapshot interface on the device cache: `state` / `meta_state`
(page "quant_kv.py") and `commit_verified_snapshot` (page "kv_cache.py"),
checked against the oracle cache: returned flags, lengths and every stored row
bit for bit, then attention over the result."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import attention, codec
from oracle.cache import OracleCache, commit_verified_snapshot as oracle_commit
from parity_util import assert_rows_equal, compare_out, f32, oracle_blocks

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rot():
    from rotated_bit_quantized_gb300 import Rotation
    return Rotation(0, 256)


@pytest.fixture(scope="module")
def mb():
    return oracle_blocks(0)


def test_state_round_trip(rot, mb):
    from rotated_bit_quantized_gb300 import IQCache
    B, H = 2, 2
    cache = IQCache(B, H)
    k, v = si.kv_tokens(81, B, H, 300, outliers=True)
    cache.append(k.cuda(), v.cuda(), rot)
    st = cache.state
    assert st[0][0].shape == (B, H, 300, 32) and st[1][0].shape == (B, H, 300, 24)
    meta = cache.meta_state
    assert meta == ("64", "4", "3")
    # the cache moves on; the state tensors do not change (copies, like the page's slices)
    k2, v2 = si.kv_tokens(81, B, H, 60, outliers=True, step=1)
    cache.trim(np.array([40, 7], dtype=np.int32))
    cache.append(k2.cuda(), v2.cuda(), rot)
    cache.state = st
    cache.meta_state = meta
    assert cache.lens.tolist() == [300, 300]
    for b in range(B):
        for h in range(H):
            assert_rows_equal(cache, b, h, 0, 300, f32(k[b, h]), f32(v[b, h]), mb)
    oc = OracleCache(B, H)
    oc.append(f32(k), f32(v), mb)
    q = si.queries(82, B, 16, 1)
    compare_out(cache.attend(q.cuda(), rot, out_dtype=torch.float32), attention.attend(f32(q), oc, mb), "after state")
    with pytest.raises(ValueError):
        cache.meta_state = ("128", "4", "3")


def test_state_of_another_format_is_adopted(rot, mb):
    from rotated_bit_quantized_gb300 import IQCache
    src = IQCache(1, 2, k_bits=2, v_bits=8, group_size=128)
    k, v = si.kv_tokens(83, 1, 2, 200, outliers=True)
    src.append(k.cuda(), v.cuda(), rot)
    dst = IQCache(1, 2)
    dst.state = src.state
    dst.meta_state = src.meta_state
    assert (dst.k_bits, dst.v_bits, dst.group_size) == (2, 8, 128) and dst.lens.tolist() == [200]
    oc = OracleCache(1, 2, k_bits=2, v_bits=8, group_size=128)
    oc.append(f32(k), f32(v), mb)
    q = si.queries(84, 1, 16, 1)
    compare_out(dst.attend(q.cuda(), rot, out_dtype=torch.float32), attention.attend(f32(q), oc, mb),
                "adopted format")


@pytest.mark.parametrize("accepted,verified,n_snaps", [(4, 4, 4), (0, 4, 4), (3, 4, 2), (1, 4, 4), (2, 4, 4),
                                                       (3, 4, 4), (4, None, 4)])
def test_commit_verified_snapshot_matches_oracle(rot, mb, accepted, verified, n_snaps):
    """Stepwise verify: append one draft token per step and snapshot; then
    commit `accepted` of the drafts, on the device cache and on the oracle."""
    from rotated_bit_quantized_gb300 import IQCache, commit_verified_snapshot
    B, H = 2, 2
    base_k, base_v = si.kv_tokens(85, B, H, 130, outliers=True)
    cache, oc = IQCache(B, H), OracleCache(B, H)
    cache.append(base_k.cuda(), base_v.cuda(), rot)
    oc.append(f32(base_k), f32(base_v), mb)
    snaps, osnaps = [], []
    for s in range(4):
        k, v = si.kv_tokens(85, B, H, 1, outliers=True, step=s)
        cache.append(k.cuda(), v.cuda(), rot)
        oc.append(f32(k), f32(v), mb)
        snaps.append(cache.snapshot())
        osnaps.append(oc.snapshot())
    got = commit_verified_snapshot(cache, snaps[:n_snaps], accepted, verified)
    want = oracle_commit(oc, osnaps[:n_snaps], accepted, verified)
    assert got == want
    assert cache.lens.tolist() == oc.lens.tolist()
    for b in range(B):
        for h in range(H):
            n = int(oc.lens[b])
            np.testing.assert_array_equal(cache.k_codes[b, h, :n].cpu().numpy().view(np.uint32), oc.k[0][b, h, :n])
            np.testing.assert_array_equal(cache.v_codes[b, h, :n].cpu().numpy().view(np.uint32), oc.v[0][b, h, :n])
            np.testing.assert_array_equal(cache.v_scales[b, h, :n].float().cpu().numpy(), oc.v[1][b, h, :n])
    q = si.queries(86, B, 16, 1)
    compare_out(cache.attend(q.cuda(), rot, out_dtype=torch.float32), attention.attend(f32(q), oc, mb),
                f"after commit {accepted}/{verified}")
    # the snapshots are intact after the commit (the restore copied them)
    if got and n_snaps:
        assert int(snaps[0].lens[0]) == 131
