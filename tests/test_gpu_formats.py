"""Cache formats other than 4-bit keys / 3-bit values / 64-dim groups (the
page's cache class takes k_bits, v_bits and group_size): CUDA path vs the CPU
oracle on the same seeded inputs.

Bars as for the tuned format: packed words, scales and biases bit-exact on
every row; attention max-abs <= 2e-3 against the oracle's unrounded output
(fp32 output), plus half a bf16 ulp for the bf16 output.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import attention, codec
from oracle.cache import OracleCache
from parity_util import cache_arrays, compare_out, f32, oracle_blocks

pytestmark = pytest.mark.gpu

# (k_bits, v_bits, group_size): every width and group size at least once
FORMATS = [(2, 2, 32), (3, 5, 128), (5, 6, 64), (8, 8, 128), (6, 3, 32), (4, 3, 32), (8, 2, 64), (4, 4, 128)]


@pytest.fixture(scope="module")
def rot():
    from rotated_bit_quantized_gb300 import Rotation
    return Rotation(0, 256)


@pytest.fixture(scope="module")
def mb():
    return oracle_blocks(0)


def assert_format_rows(cache, b, h, lo, hi, k_rows, v_rows, mb, kb, vb, gs):
    kw, ks, kbias = codec.encode_rows(k_rows, mb, kb, gs)
    vw, vs, vbias = codec.encode_rows(v_rows, mb, vb, gs)
    got = cache_arrays(cache, b, h, hi)
    names = ("k_codes", "k_scales", "k_biases", "v_codes", "v_scales", "v_biases")
    for name, g, w in zip(names, got, (kw, ks, kbias, vw, vs, vbias)):
        g = g[lo:hi]
        assert g.shape == w.shape, (name, g.shape, w.shape)
        if g.dtype == np.uint32:
            bad = np.count_nonzero(g != w)
            assert bad == 0, f"{name} ({b},{h}) rows {lo}:{hi} k{kb}v{vb}g{gs}: {bad} words differ"
        else:
            np.testing.assert_array_equal(g, w, err_msg=f"{name} ({b},{h}) k{kb}v{vb}g{gs}")


def build_pair(rot, mb, B, H, T, fmt, seed, trims=None, then_append=0):
    from rotated_bit_quantized_gb300 import IQCache
    kb, vb, gs = fmt
    cache = IQCache(B, H, k_bits=kb, v_bits=vb, group_size=gs)
    oc = OracleCache(B, H, k_bits=kb, v_bits=vb, group_size=gs)
    k, v = si.kv_tokens(seed, B, H, T, outliers=True)
    cache.reserve(T + then_append + 256)
    cache.append(k.cuda(), v.cuda(), rot)
    oc.append(f32(k), f32(v), mb)
    if trims is not None:
        cache.trim(np.array(trims))
        oc.trim(np.array(trims))
    if then_append:
        k2, v2 = si.kv_tokens(seed, B, H, then_append, outliers=True, step=0)
        cache.append(k2.cuda(), v2.cuda(), rot)
        oc.append(f32(k2), f32(v2), mb)
    torch.cuda.synchronize()
    return cache, oc


@pytest.mark.parametrize("fmt", FORMATS)
def test_append_bit_exact(rot, mb, fmt):
    """Rows of two appends (the second at a ragged offset), then a trim and a
    third append over the trimmed rows: every row bit-exact."""
    from rotated_bit_quantized_gb300 import IQCache
    kb, vb, gs = fmt
    B, H = 2, 2
    cache = IQCache(B, H, k_bits=kb, v_bits=vb, group_size=gs)
    rows = {(b, h): ([], []) for b in range(B) for h in range(H)}
    for step, (op, arg) in enumerate([("a", 200), ("a", 37), ("t", [9, 0]), ("a", 300)]):
        if op == "a":
            k, v = si.kv_tokens(70 + kb, B, H, arg, outliers=True, step=step)
            cache.append(k.cuda(), v.cuda(), rot)
            for b in range(B):
                for h in range(H):
                    rows[(b, h)][0].extend(f32(k[b, h]))
                    rows[(b, h)][1].extend(f32(v[b, h]))
        else:
            t = cache.trim(np.array(arg))
            for b in range(B):
                for h in range(H):
                    for lst in rows[(b, h)]:
                        del lst[len(lst) - t[b]:]
    torch.cuda.synchronize()
    for b in range(B):
        for h in range(H):
            n = int(cache.lens[b])
            assert_format_rows(cache, b, h, 0, n, np.array(rows[(b, h)][0]), np.array(rows[(b, h)][1]),
                               mb, kb, vb, gs)


ATTEND_CASES = [
    # B, Hkv, rep, T, L, causal, trims
    (2, 2, 8, 1500, 1, False, [0, 41]),
    (1, 2, 8, 700, 4, True, None),
    (2, 1, 4, 333, 3, True, [5, 0]),
]


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("B,H,rep,T,L,causal,trims", ATTEND_CASES)
def test_attend_matches_oracle(rot, mb, fmt, B, H, rep, T, L, causal, trims):
    cache, oc = build_pair(rot, mb, B, H, T, fmt, seed=80 + T, trims=trims, then_append=L if causal else 0)
    q = si.queries(81 + T, B, H * rep, L)
    ref = attention.attend(f32(q), oc, mb, causal=causal)
    for dt in (torch.float32, torch.bfloat16):
        out = cache.attend(q.cuda(), rot, causal=causal, out_dtype=dt)
        torch.cuda.synchronize()
        compare_out(out, ref, f"{fmt} B{B} H{H} rep{rep} T{T} L{L} causal{causal} {dt}")
    assert cache.device_status() == 0


@pytest.mark.parametrize("fmt", [(2, 2, 32), (8, 8, 128)])
@pytest.mark.parametrize("kind", ["bool", "add"])
def test_explicit_masks(rot, mb, fmt, kind):
    B, H, rep, T, L = 2, 2, 8, 600, 2
    cache, oc = build_pair(rot, mb, B, H, T, fmt, seed=90)
    rng = np.random.default_rng(91)
    keep = rng.random((B, L, T)) < 0.7
    keep[:, :, -1] = True
    if kind == "bool":
        mask = keep
    else:
        mask = np.where(keep, rng.standard_normal((B, L, T)).astype(np.float32), -np.inf).astype(np.float32)
    q = si.queries(92, B, H * rep, L)
    ref = attention.attend(f32(q), oc, mb, mask=mask)
    out = cache.attend(q.cuda(), rot, mask=torch.from_numpy(mask).cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    compare_out(out, ref, f"{fmt} {kind} mask")
    assert cache.device_status() == 0


@pytest.mark.parametrize("fmt", [(3, 5, 128), (6, 3, 32)])
def test_decode_step_snapshot_restore(rot, mb, fmt):
    """append_attend (append then attend for these formats), snapshot,
    further steps, restore: the restored cache equals the snapshot row for row
    and attends like the oracle at that point."""
    kb, vb, gs = fmt
    B, H, rep = 2, 2, 8
    cache, oc = build_pair(rot, mb, B, H, 400, fmt, seed=95)
    for s in range(3):
        k, v = si.kv_tokens(95, B, H, 1, outliers=True, step=s + 1)
        q = si.queries(96, B, H * rep, 1, step=s)
        out = cache.append_attend(k.cuda(), v.cuda(), q.cuda(), rot, out_dtype=torch.float32)
        oc.append(f32(k), f32(v), mb)
        ref = attention.attend(f32(q), oc, mb)
        torch.cuda.synchronize()
        compare_out(out, ref, f"{fmt} decode step {s}")
    snap = cache.snapshot()
    osnap = oc.snapshot()
    k, v = si.kv_tokens(95, B, H, 7, outliers=True, step=9)
    cache.append(k.cuda(), v.cuda(), rot)
    cache.restore(snap)
    oc.restore(osnap)
    torch.cuda.synchronize()
    assert cache.lens.tolist() == [int(x) for x in oc.lens]
    q = si.queries(97, B, H * rep, 1)
    ref = attention.attend(f32(q), oc, mb)
    out = cache.attend(q.cuda(), rot, out_dtype=torch.float32)
    torch.cuda.synchronize()
    compare_out(out, ref, f"{fmt} after restore")
    assert cache.device_status() == 0
