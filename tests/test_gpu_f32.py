"""float32 caches (float32 keys, values and queries; float32 scales and
biases, as the page's `_init_quant(..., dt)` stores them for float32 keys;
the float32 rotation blocks, as `rotate_last` casts M to float32): the CUDA
path against the oracle's float32 path on the same seeded float32 inputs.

Bars: packed words, scales and biases bit-exact on every row; attention
max-abs <= ATOL_F32 = 2e-5 on the float32 output against the oracle's
unrounded output, plus half a bf16 ulp for the bf16 output.  The oracle
rounds q' and q'' to float32 like the kernel and carries everything after
that in float64, so the difference is the kernel's own float32 arithmetic:
256-term score sums, one rounding per dequantised element, the
2^-22-relative exp2 approximation and float32 P.V sums over up to 1500 keys.
Each contributes relative errors of order 1e-6 on outputs of order 1 (the
largest difference measured over the cases below is 4.1e-6); the bar leaves
a factor of about 5.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import attention, bf16, codec, rotation
from oracle.cache import OracleCache
from parity_util import compare_out, f32

pytestmark = pytest.mark.gpu

ATOL_F32 = 2e-5
FORMATS = [(4, 3, 64), (2, 2, 32), (8, 8, 128), (3, 5, 128)]


@pytest.fixture(scope="module")
def rot():
    from rotated_bit_quantized_gb300 import Rotation
    return Rotation(0, 256)


@pytest.fixture(scope="module")
def m32():
    return rotation.build_blocks(si.rotation_draws(0, 256))


def device_rows(cache, b, h, n):
    kw = cache.k_codes[b, h, :n].cpu().numpy().view(np.uint32)
    vw = cache.v_codes[b, h, :n].cpu().numpy().view(np.uint32)
    meta = [getattr(cache, name)[b, h, :n].cpu().numpy() for name in ("k_scales", "k_biases", "v_scales", "v_biases")]
    return kw, meta[0], meta[1], vw, meta[2], meta[3]


def assert_f32_rows(cache, b, h, lo, hi, k_rows, v_rows, m32, kb, vb, gs):
    kw, ks, kbias = codec.encode_rows(k_rows, m32, kb, gs, dtype="f32")
    vw, vs, vbias = codec.encode_rows(v_rows, m32, vb, gs, dtype="f32")
    got = device_rows(cache, b, h, hi)
    names = ("k_codes", "k_scales", "k_biases", "v_codes", "v_scales", "v_biases")
    for name, g, w in zip(names, got, (kw, ks, kbias, vw, vs, vbias)):
        g = g[lo:hi]
        assert g.shape == w.shape, (name, g.shape, w.shape)
        if g.dtype == np.uint32:
            bad = np.count_nonzero(g != w)
            assert bad == 0, f"{name} ({b},{h}) rows {lo}:{hi} k{kb}v{vb}g{gs}: {bad} words differ"
        else:
            assert g.dtype == np.float32
            np.testing.assert_array_equal(g.view(np.uint32), w.astype(np.float32).view(np.uint32),
                                          err_msg=f"{name} ({b},{h}) k{kb}v{vb}g{gs}")


def build_pair(rot, m32, B, H, T, fmt, seed, trims=None, then_append=0):
    from rotated_bit_quantized_gb300 import IQCache
    kb, vb, gs = fmt
    cache = IQCache(B, H, k_bits=kb, v_bits=vb, group_size=gs, dtype=torch.float32)
    oc = OracleCache(B, H, k_bits=kb, v_bits=vb, group_size=gs, dtype="f32")
    k, v = si.kv_tokens(seed, B, H, T, outliers=True, dtype=torch.float32)
    cache.reserve(T + then_append + 256)
    cache.append(k.cuda(), v.cuda(), rot)
    oc.append(f32(k), f32(v), m32)
    if trims is not None:
        cache.trim(np.array(trims))
        oc.trim(np.array(trims))
    if then_append:
        k2, v2 = si.kv_tokens(seed, B, H, then_append, outliers=True, step=0, dtype=torch.float32)
        cache.append(k2.cuda(), v2.cuda(), rot)
        oc.append(f32(k2), f32(v2), m32)
    torch.cuda.synchronize()
    return cache, oc


@pytest.mark.parametrize("fmt", FORMATS)
def test_f32_append_bit_exact(rot, m32, fmt):
    """Two appends (the second at a ragged offset), a trim and a third append
    over the trimmed rows: every row's words, float32 scales and float32
    biases bit-exact."""
    from rotated_bit_quantized_gb300 import IQCache
    kb, vb, gs = fmt
    B, H = 2, 2
    cache = IQCache(B, H, k_bits=kb, v_bits=vb, group_size=gs, dtype=torch.float32)
    assert cache.k_scales.dtype == torch.float32 and cache.v_biases.dtype == torch.float32
    rows = {(b, h): ([], []) for b in range(B) for h in range(H)}
    for step, (op, arg) in enumerate([("a", 200), ("a", 37), ("t", [9, 0]), ("a", 300)]):
        if op == "a":
            k, v = si.kv_tokens(170 + kb, B, H, arg, outliers=True, step=step, dtype=torch.float32)
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
            assert_f32_rows(cache, b, h, 0, n, np.array(rows[(b, h)][0]), np.array(rows[(b, h)][1]),
                            m32, kb, vb, gs)
    # float32 metadata, not bfloat16 values in float32 slots
    s = cache.k_scales[:, :, :200].cpu().numpy()
    assert np.mean(bf16.round_bf16(s) == s) < 0.1


def test_f32_append_special_rows(rot, m32):
    """Constant groups (scale 0, all codes 0), huge and tiny magnitudes, and
    values that are not bfloat16 numbers: bit-exact against the oracle."""
    from rotated_bit_quantized_gb300 import IQCache
    cache = IQCache(1, 1, dtype=torch.float32)
    rng = np.random.default_rng(5)
    k = rng.standard_normal((1, 1, 6, 256)).astype(np.float32)
    k[0, 0, 0] = 1.2345678
    k[0, 0, 1, :64] = -3.0e30
    k[0, 0, 1, 64:] *= np.float32(1e30)
    k[0, 0, 2] *= np.float32(1e-30)
    k[0, 0, 3] = np.float32(1.0) + np.arange(256, dtype=np.float32) * np.float32(2.0 ** -20)
    k[0, 0, 4] = 0.0
    v = k[:, :, ::-1].copy()
    cache.append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), rot)
    torch.cuda.synchronize()
    assert_f32_rows(cache, 0, 0, 0, 6, k[0, 0], v[0, 0], m32, 4, 3, 64)


ATTEND_CASES = [
    # B, Hkv, rep, T, L, causal, trims
    (2, 2, 8, 1500, 1, False, [0, 41]),
    (1, 2, 8, 700, 4, True, None),
    (2, 1, 4, 333, 3, True, [5, 0]),
]


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("B,H,rep,T,L,causal,trims", ATTEND_CASES)
def test_f32_attend_matches_oracle(rot, m32, fmt, B, H, rep, T, L, causal, trims):
    cache, oc = build_pair(rot, m32, B, H, T, fmt, seed=180 + T, trims=trims, then_append=L if causal else 0)
    q = si.queries(181 + T, B, H * rep, L, dtype=torch.float32)
    ref = attention.attend(f32(q), oc, m32, causal=causal)
    out = cache.attend(q.cuda(), rot, causal=causal)
    assert out.dtype == torch.float32  # the queries' dtype by default, as the page returns
    torch.cuda.synchronize()
    err = compare_out(out, ref, f"f32 {fmt} B{B} H{H} rep{rep} T{T} L{L} causal{causal}", atol=ATOL_F32)
    print(f"f32 {fmt} B{B} rep{rep} T{T} L{L}: max abs err {err:.2e}")
    outb = cache.attend(q.cuda(), rot, causal=causal, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    compare_out(outb, ref, f"f32 {fmt} bf16 output", atol=ATOL_F32)
    assert cache.device_status() == 0


@pytest.mark.parametrize("kind", ["bool", "add"])
def test_f32_explicit_masks(rot, m32, kind):
    B, H, rep, T, L = 2, 2, 8, 600, 2
    cache, oc = build_pair(rot, m32, B, H, T, (4, 3, 64), seed=190)
    rng = np.random.default_rng(191)
    keep = rng.random((B, L, T)) < 0.7
    keep[:, :, -1] = True
    if kind == "bool":
        mask = keep
        mask[1, 1, :] = False  # every key masked: the uniform mean, as the page's softmax gives
    else:
        mask = np.where(keep, rng.standard_normal((B, L, T)).astype(np.float32), -np.inf).astype(np.float32)
    q = si.queries(192, B, H * rep, L, dtype=torch.float32)
    ref = attention.attend(f32(q), oc, m32, mask=mask)
    out = cache.attend(q.cuda(), rot, mask=torch.from_numpy(mask).cuda())
    torch.cuda.synchronize()
    compare_out(out, ref, f"f32 {kind} mask", atol=ATOL_F32)
    assert cache.device_status() == 0


def test_f32_decode_steps_grow_snapshot_restore(rot, m32):
    """append_attend steps across a capacity growth, then snapshot, more steps
    and restore: rows bit-exact, attention as the oracle at every point."""
    B, H, rep = 2, 2, 8
    cache, oc = build_pair(rot, m32, B, H, 250, (4, 3, 64), seed=195)
    cap0 = cache.capacity
    for s in range(12):  # 250 + 12 rows cross the first 256-row boundary
        k, v = si.kv_tokens(195, B, H, 1, outliers=True, step=s + 1, dtype=torch.float32)
        q = si.queries(196, B, H * rep, 1, step=s, dtype=torch.float32)
        out = cache.append_attend(k.cuda(), v.cuda(), q.cuda(), rot, causal=True)
        oc.append(f32(k), f32(v), m32)
        ref = attention.attend(f32(q), oc, m32, causal=True)
        torch.cuda.synchronize()
        compare_out(out, ref, f"f32 decode step {s}", atol=ATOL_F32)
    assert cache.capacity > cap0 or cap0 >= 262
    snap = cache.snapshot()
    osnap = oc.snapshot()
    k, v = si.kv_tokens(195, B, H, 7, outliers=True, step=99, dtype=torch.float32)
    cache.append(k.cuda(), v.cuda(), rot)
    cache.restore(snap)
    oc.restore(osnap)
    torch.cuda.synchronize()
    assert cache.lens.tolist() == [int(x) for x in oc.lens]
    for b in range(B):
        for h in range(H):
            n = int(cache.lens[b])
            got = device_rows(cache, b, h, n)
            for g, w in zip(got, (oc.k[0], oc.k[1], oc.k[2], oc.v[0], oc.v[1], oc.v[2])):
                assert np.array_equal(g, w[b, h, :n])
    q = si.queries(197, B, H * rep, 1, dtype=torch.float32)
    ref = attention.attend(f32(q), oc, m32)
    out = cache.attend(q.cuda(), rot)
    torch.cuda.synchronize()
    compare_out(out, ref, "f32 after restore", atol=ATOL_F32)
    st = cache.state
    assert st[0][1].dtype == torch.float32
    assert cache.device_status() == 0


def test_f32_rejects_mismatched_dtypes(rot):
    from rotated_bit_quantized_gb300 import IQCache
    cache = IQCache(1, 2, dtype=torch.float32)
    kb, vb = si.kv_tokens(1, 1, 2, 4)  # bfloat16 data into a float32 cache
    with pytest.raises(ValueError):
        cache.append(kb.cuda(), vb.cuda(), rot)
    k, v = si.kv_tokens(1, 1, 2, 4, dtype=torch.float32)
    cache.append(k.cuda(), v.cuda(), rot)
    with pytest.raises(ValueError):
        cache.attend(si.queries(1, 1, 16, 1).cuda(), rot)
    bf = IQCache(1, 2)
    with pytest.raises(ValueError):
        bf.append(k.cuda(), v.cuda(), rot)
