"""CUDA path vs the CPU oracle, element by element, on small seeded inputs that
span several 64-token tiles, several key chunks and ragged tails.

Bars: rotation blocks, packed words, scales and biases bit-exact; attention
max-abs <= 2e-3 against the oracle's unrounded output (fp32 output), plus half
a bf16 ulp for the bf16 output.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import attention, bf16, rotation
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


@pytest.mark.parametrize("seed", [0, 1, 5, 123])
def test_rotation_bit_exact(seed):
    from rotated_bit_quantized_gb300 import Rotation
    r = Rotation(seed, 256)
    want = rotation.build_blocks(si.rotation_draws(seed, 256))
    got = r.blocks_f32.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    gotb = r.blocks_bf16.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(gotb, bf16.f32_to_bf16_bits(want))


def test_append_trim_append_bit_exact(rot, mb):
    from rotated_bit_quantized_gb300 import IQCache
    B, H = 2, 2
    cache = IQCache(B, H)
    rows = {(b, h): ([], []) for b in range(B) for h in range(H)}
    plan = [("a", 300), ("a", 1), ("t", [5, 0]), ("a", 77), ("t", [400, 13]), ("a", 40)]
    for step, (op, arg) in enumerate(plan):
        if op == "a":
            k, v = si.kv_tokens(9, B, H, arg, outliers=True, step=step)
            cache.append(k.cuda(), v.cuda(), rot)
            for b in range(B):
                for h in range(H):
                    rows[(b, h)][0].extend(f32(k[b, h]))
                    rows[(b, h)][1].extend(f32(v[b, h]))
        else:
            t = cache.trim(np.array(arg))
            for b in range(B):
                assert t[b] == min(arg[b], len(rows[(b, 0)][0]))
                for h in range(H):
                    for lst in rows[(b, h)]:
                        del lst[len(lst) - t[b]:]
        torch.cuda.synchronize()
        for b in range(B):
            assert cache.lens[b] == len(rows[(b, 0)][0])
            for h in range(H):
                n = int(cache.lens[b])
                if n:
                    assert_rows_equal(cache, b, h, 0, n, np.array(rows[(b, h)][0]),
                                      np.array(rows[(b, h)][1]), mb)
    assert cache.capacity % 256 == 0


def test_append_special_groups(rot, mb):
    """Constant groups (scale 0), huge and tiny magnitudes, exact ties of the
    quantiser: all bit-exact."""
    from rotated_bit_quantized_gb300 import IQCache
    rng = np.random.default_rng(3)
    n = 64
    k = rng.standard_normal((1, 1, n, 256)).astype(np.float32)
    k[0, 0, 0] = 1.0                       # constant row before rotation
    k[0, 0, 1] = 0.0                       # all zeros -> every group constant
    k[0, 0, 2] *= 1e30
    k[0, 0, 3] *= 1e-30
    k[0, 0, 4] = np.round(k[0, 0, 4] * 4) / 4
    v = k[:, :, ::-1].copy()
    kt, vt = si.to_bf16(k), si.to_bf16(v)
    cache = IQCache(1, 1)
    cache.append(kt.cuda(), vt.cuda(), rot)
    torch.cuda.synchronize()
    assert_rows_equal(cache, 0, 0, 0, n, f32(kt[0, 0]), f32(vt[0, 0]), mb)


def build_pair(rot, mb, B, H, T, seed, outliers=True, trims=None, then_append=0):
    """Device cache and oracle cache holding the same tokens."""
    from rotated_bit_quantized_gb300 import IQCache
    cache = IQCache(B, H)
    oc = OracleCache(B, H)
    k, v = si.kv_tokens(seed, B, H, T, outliers=outliers)
    cache.append(k.cuda(), v.cuda(), rot)
    oc.append(f32(k), f32(v), mb)
    if trims is not None:
        cache.trim(np.array(trims))
        oc.trim(np.array(trims))
    if then_append:
        k, v = si.kv_tokens(seed, B, H, then_append, outliers=outliers, step=0)
        cache.append(k.cuda(), v.cuda(), rot)
        oc.append(f32(k), f32(v), mb)
    return cache, oc


CASES = [
    # B, Hkv, rep, T, L, causal, trims
    (1, 1, 1, 256, 1, False, None),
    (2, 2, 8, 300, 1, False, None),
    (2, 2, 8, 1000, 1, True, [0, 37]),
    (3, 2, 8, 777, 4, True, [0, 3, 64]),
    (1, 2, 8, 333, 3, True, None),
    (1, 2, 4, 500, 2, False, None),
    (1, 1, 2, 130, 1, False, None),
    (2, 1, 8, 20, 1, False, None),
    (1, 2, 8, 600, 64, True, None),
    (1, 1, 8, 5000, 1, False, None),
    # >= 128 query rows per kv head: the tensor-memory prefill kernel
    (1, 2, 8, 700, 20, True, None),      # 160 rows: a full and a ragged row tile
    (2, 1, 4, 900, 40, False, [0, 130]),  # rep 4, no mask, ragged lengths
    (1, 2, 2, 1100, 100, True, None),    # rep 2, 200 rows
]


@pytest.mark.parametrize("B,H,rep,T,L,causal,trims", CASES)
def test_attend_matches_oracle(rot, mb, B, H, rep, T, L, causal, trims):
    cache, oc = build_pair(rot, mb, B, H, T, seed=11 + T, trims=trims, then_append=L if causal else 0)
    q = si.queries(12 + T, B, H * rep, L)
    ref = attention.attend(f32(q), oc, mb, causal=causal)
    for dt in (torch.float32, torch.bfloat16):
        out = cache.attend(q.cuda(), rot, causal=causal, out_dtype=dt)
        torch.cuda.synchronize()
        compare_out(out, ref, f"B{B} H{H} rep{rep} T{T} L{L} causal{causal} {dt}")
    assert cache.device_status() == 0


def test_stale_rows_are_never_read(rot, mb):
    cache, oc = build_pair(rot, mb, 2, 2, 700, seed=21, trims=[100, 7])
    q = si.queries(22, 2, 16, 1).cuda()
    ref = cache.attend(q, rot, out_dtype=torch.float32).clone()
    for b in range(2):
        n = int(cache.lens[b])
        for name in ("k_scales", "k_biases", "v_scales", "v_biases"):
            getattr(cache, name)[b, :, n:] = float("nan")
        cache.k_codes[b, :, n:] = -1
        cache.v_codes[b, :, n:] = -1
    out = cache.attend(q, rot, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    compare_out(out, attention.attend(f32(q.cpu()), oc, mb), "stale rows")


def test_repeated_calls_are_deterministic(rot, mb):
    cache, _ = build_pair(rot, mb, 2, 2, 3000, seed=31)
    q = si.queries(32, 2, 16, 4).cuda()
    a = cache.attend(q, rot, causal=True, out_dtype=torch.float32).clone()
    b = cache.attend(q, rot, causal=True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_gather_snapshot_tile_keep_row(rot, mb):
    from rotated_bit_quantized_gb300 import IQCache
    cache, oc = build_pair(rot, mb, 1, 2, 300, seed=41)
    snap = cache.snapshot()
    k, v = si.kv_tokens(41, 1, 2, 10, outliers=True, step=3)
    cache.trim(5)
    cache.append(k.cuda(), v.cuda(), rot)
    cache.restore(snap)
    torch.cuda.synchronize()
    assert cache.lens.tolist() == [300]
    kk, vv = si.kv_tokens(41, 1, 2, 300, outliers=True)
    for h in range(2):
        assert_rows_equal(cache, 0, h, 0, 300, f32(kk[0, h]), f32(vv[0, h]), mb)
    cache.tile(3)
    cache.commit_verified_prefix(4, np.array([4, 1, 2]))
    assert cache.lens.tolist() == [300, 297, 298]
    cache.keep_row(2)
    torch.cuda.synchronize()
    assert cache.batch == 1 and cache.lens.tolist() == [298]
    for h in range(2):
        assert_rows_equal(cache, 0, h, 0, 298, f32(kk[0, h, :298]), f32(vv[0, h, :298]), mb)
    with pytest.raises(ValueError):
        cache.commit_verified_prefix(4, 5)
    big = IQCache(1, 2, capacity=256)
    big.reserve(1000)
    assert big.capacity == 1024
