"""Pins of the oracle's bf16 rounding, rotation and codec against things other than itself.

Closed forms, textbook routines, brute force and hand-worked fixtures
(tests/golden/).  CPU only.
"""
import json
import os

import numpy as np
import pytest

from oracle import bf16, codec, rotation
import seeded_inputs as si

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- bf16

def _bf16_candidates(x):
    """The two bf16 neighbours of float32 x, found by truncation and +1 ulp."""
    u = np.float32(x).view(np.uint32)
    lo = np.uint32(u & np.uint32(0xFFFF0000))
    hi = np.uint32(lo + np.uint32(0x10000))
    return lo.view(np.float32), hi.view(np.float32)


def test_ulp_bf16_is_the_gap_to_the_next_bf16():
    """ulp_bf16(x) (the output tolerance's bf16 term) equals the distance from
    the bf16 value at or below |x| to the next one, found on the bit pattern
    (+1 in the 16-bit representation): normals, powers of two (the gap above),
    the subnormal range (a fixed 2^-133) and zero."""
    rng = np.random.default_rng(5)
    mags = np.concatenate([
        np.exp(rng.uniform(np.log(2.0 ** -125), np.log(2.0 ** 120), 4000)),  # normals, anywhere in range
        2.0 ** np.arange(-126, 127, dtype=np.float64),                          # exact powers of two
        rng.uniform(0, 2.0 ** -126, 200),                                       # subnormal range
        [0.0, 1.0, 1.5, 3.0, 255.0, 256.0, 65504.0]])
    xs = np.concatenate([mags, -mags]).astype(np.float32)
    for x in xs:
        lo, hi = _bf16_candidates(abs(x))  # truncation: the bf16 at or below |x|, and the next one
        gap = float(hi) - float(lo)
        assert bf16.ulp_bf16(x) == gap, (x, bf16.ulp_bf16(x), gap)


def test_bf16_is_nearest_with_ties_to_even():
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 10,
                         np.float32([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 2.0 ** -130])])
    r = bf16.round_bf16(xs)
    for x, y in zip(xs, r):
        lo, hi = _bf16_candidates(x)
        dlo, dhi = abs(float(x) - float(lo)), abs(float(x) - float(hi))
        if dlo < dhi:
            assert y == lo
        elif dhi < dlo:
            assert y == hi
        else:  # tie: the even mantissa (bit 16 clear)
            even = lo if (lo.view(np.uint32) >> 16) % 2 == 0 else hi
            assert y == even


def test_bf16_hand_values():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1.0 (0x3F80)
    assert bf16.f32_to_bf16_bits(np.float32(1 + 2 ** -8)) == 0x3F80
    # 1 + 3*2^-8 is halfway between 1+2^-7 (odd) and 1+2^-6 (even) -> 0x3F82
    assert bf16.f32_to_bf16_bits(np.float32(1 + 3 * 2 ** -8)) == 0x3F82
    assert bf16.f32_to_bf16_bits(np.float32(-2.0)) == 0xC000
    assert bf16.f32_to_bf16_bits(np.float32(np.inf)) == 0x7F80
    assert np.isnan(bf16.round_bf16(np.float32(np.nan)))
    # the largest float32 rounds up to infinity
    assert bf16.f32_to_bf16_bits(np.float32(3.4028235e38)) == 0x7F80


# ---------------------------------------------------------------- rotation

def hamilton(p, q):
    """Textbook quaternion product p*q, (w, x, y, z) convention."""
    a1, b1, c1, d1 = p
    a2, b2, c2, d2 = q
    return np.array([a1 * a2 - b1 * b2 - c1 * c2 - d1 * d2,
                     a1 * b2 + b1 * a2 + c1 * d2 - d1 * c2,
                     a1 * c2 - b1 * d2 + c1 * a2 + d1 * b2,
                     a1 * d2 + b1 * c2 - c1 * b2 + d1 * a2])


def conj(q):
    return np.array([q[0], -q[1], -q[2], -q[3]])


def test_quat_left_is_hamilton_left_multiplication():
    rng = np.random.default_rng(1)
    for _ in range(50):
        q, v = rng.standard_normal(4), rng.standard_normal(4)
        np.testing.assert_allclose(rotation.quat_left(q) @ v, hamilton(q, v), atol=1e-12)


def test_printed_right_conj_matrix_is_left_multiplication_by_conjugate():
    # The printed matrix maps v -> conj(q)*v (it is L(q)^T), not v -> v*conj(q).
    rng = np.random.default_rng(2)
    q = rng.standard_normal(4)
    q /= np.linalg.norm(q)
    for _ in range(20):
        v = rng.standard_normal(4)
        np.testing.assert_allclose(rotation.quat_right_conj(q) @ v, hamilton(conj(q), v), atol=1e-12)
    v = rng.standard_normal(4)
    assert not np.allclose(rotation.quat_right_conj(q) @ v, hamilton(v, conj(q)))


def test_normalize_f32_close_to_exact_unit_vector():
    rng = np.random.default_rng(3)
    for _ in range(200):
        v = rng.standard_normal(4).astype(np.float32)
        q = rotation.normalize_f32(v).astype(np.float64)
        exact = v.astype(np.float64) / np.linalg.norm(v.astype(np.float64))
        np.testing.assert_allclose(q, exact, rtol=4e-7, atol=1e-7)


def test_golden_rotation_blocks():
    for case in load("rotation_blocks.json")["cases"]:
        draws = np.array([[case["qL"], case["qR"]]], dtype=np.float32)
        got = rotation.build_blocks(draws)[0]
        want = np.array([[np.float32(float(e)) for e in row] for row in case["block"]], dtype=np.float32)
        np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("seed", [0, 1, 17])
def test_rotation_orthogonal_det_one_block_diagonal(seed):
    blocks = rotation.build_blocks(si.rotation_draws(seed, 256))
    m = rotation.dense(blocks)
    np.testing.assert_allclose(m @ m.T, np.eye(256), atol=1e-6)
    for b in range(64):
        assert abs(np.linalg.det(blocks[b].astype(np.float64)) - 1.0) < 1e-6
    mask = np.kron(np.eye(64), np.ones((4, 4))) == 0
    assert (m[mask] == 0).all()


def test_block_equals_left_isoclinic_quaternion():
    draws = si.rotation_draws(0, 256)
    blocks = rotation.build_blocks(draws)
    for b in range(64):
        ql = draws[b, 0].astype(np.float64)
        qr = draws[b, 1].astype(np.float64)
        ql, qr = ql / np.linalg.norm(ql), qr / np.linalg.norm(qr)
        p = hamilton(ql, conj(qr))
        np.testing.assert_allclose(blocks[b], rotation.quat_left(p), atol=2e-7)


def test_same_seed_same_rotation():
    a = rotation.build_blocks(si.rotation_draws(0, 256))
    b = rotation.build_blocks(si.rotation_draws(0, 256))
    c = rotation.build_blocks(si.rotation_draws(1, 256))
    np.testing.assert_array_equal(a, b)
    assert not np.array_equal(a, c)


def test_rotation_cancels_in_scores_and_inverts_on_values():
    rng = np.random.default_rng(4)
    m = rotation.dense(rotation.build_blocks(si.rotation_draws(0, 256)))
    q, k, v = rng.standard_normal((3, 256))
    assert abs((q @ m) @ (k @ m) - q @ k) < 1e-6 * (np.abs(q) @ np.abs(k))
    np.testing.assert_allclose((v @ m) @ m.T, v, atol=1e-6)


def test_rotate_matches_exact_product_rounded():
    rng = np.random.default_rng(5)
    mb = rotation.blocks_bf16(rotation.build_blocks(si.rotation_draws(0, 256)))
    x = bf16.round_bf16(rng.standard_normal((64, 256)).astype(np.float32) * 3)
    got = codec.rotate(x, mb)
    exact = x.astype(np.float64) @ rotation.dense(mb)
    # float32 ordered summation of exact products then one bf16 rounding:
    # within one bf16 ulp of the exact value, and equal to its rounding almost always
    assert np.all(np.abs(got - exact) <= bf16.ulp_bf16(exact) * 1.0 + 1e-30)
    same = np.mean(got == bf16.round_bf16(exact.astype(np.float32)))
    assert same > 0.999


# ---------------------------------------------------------------- pack / unpack

def bigint_pack(codes, bits):
    total = 0
    for i, c in enumerate(codes):
        total |= int(c) << (i * bits)
    n = len(codes) * bits // 32
    return [(total >> (32 * w)) & 0xFFFFFFFF for w in range(n)]


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_pack_matches_bigint_and_roundtrips(bits):
    rng = np.random.default_rng(bits)
    rows = [rng.integers(0, 2 ** bits, 256), np.zeros(256, int), np.full(256, 2 ** bits - 1),
            np.arange(256) % 2 * (2 ** bits - 1)]
    for r in rows:
        words = codec.pack(r[None], bits)[0]
        assert words.shape == (codec.packed_words(256, bits),)
        assert [int(w) for w in words] == bigint_pack(r, bits)
        np.testing.assert_array_equal(codec.unpack(words[None], bits, 256)[0], r)


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_packed_words_count(bits):
    assert codec.packed_words(256, bits) * 32 == 256 * bits


def test_golden_pack_examples():
    for ex in load("pack_examples.json")["examples"]:
        words = codec.pack(np.array(ex["codes"])[None], ex["bits"])[0]
        assert [int(w) for w in words] == [int(w, 16) for w in ex["words"]], ex["derivation"]


# ---------------------------------------------------------------- quantise

@pytest.mark.parametrize("name", ["quantize_4bit_ramp.json", "quantize_3bit_ties.json"])
def test_golden_quantize(name):
    g = load(name)
    x = np.array(g["values"], dtype=np.float32)[None]
    codes, s, b = codec.quantize(x, g["bits"], g["group_size"])
    assert s[0, 0] == np.float32(g["s_hat"]) and b[0, 0] == np.float32(g["b_hat"])
    assert codes[0].tolist() == g["codes"]


@pytest.mark.parametrize("gs", [32, 64, 128])
@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_quantize_error_bound_and_extremes(bits, gs):
    rng = np.random.default_rng(10 + bits + gs)
    x = bf16.round_bf16(rng.standard_normal((500, 256)).astype(np.float32) * rng.uniform(0.1, 30, (500, 1)))
    codes, s, b = codec.quantize(x, bits, gs)
    assert s.shape == b.shape == (500, 256 // gs)
    deq = codec.dequantize(codes, s, b, gs)
    # groups are runs of gs consecutive dims
    g = x.reshape(500, 256 // gs, gs).astype(np.float64)
    scale = (g.max(-1) - g.min(-1)) / (2 ** bits - 1)
    bound = s / 2 + (2 ** bits - 1) * np.abs(scale - s) + 1e-6 * np.abs(g).max(-1)
    err = np.abs(deq.reshape(500, 256 // gs, gs) - g)
    assert (err <= bound[..., None]).all()
    cg = codes.reshape(500, 256 // gs, gs)
    amin = g.argmin(-1)
    amax = g.argmax(-1)
    assert (np.take_along_axis(cg, amin[..., None], -1) == 0).all()
    top = np.take_along_axis(cg, amax[..., None], -1)
    assert (top >= 2 ** bits - 2).all()


@pytest.mark.parametrize("gs", [32, 64, 128])
def test_quantize_brute_force_nearest_level(gs):
    rng = np.random.default_rng(20 + gs)
    x = bf16.round_bf16(rng.standard_normal((300, gs)).astype(np.float32))
    for bits in (2, 3, 4, 5, 6, 8):
        codes, s, b = codec.quantize(x, bits, gs)
        levels = s[:, :, None].astype(np.float64) * np.arange(2 ** bits) + b[:, :, None]
        dist = np.abs(x.astype(np.float64)[:, :, None] - levels[:, 0][:, None, :])
        best = dist.min(-1)
        mine = np.take_along_axis(dist, codes.astype(int)[..., None], -1)[..., 0]
        # the chosen level is a nearest one up to float32 rounding of the ratio
        assert np.all(mine - best <= 1e-6 * (1 + np.abs(x)))


def test_constant_group_gives_zero_codes_and_exact_dequant():
    x = np.full((1, 64), np.float32(1.5))
    codes, s, b = codec.quantize(x, 3, 64)
    assert s[0, 0] == 0 and b[0, 0] == np.float32(1.5) and (codes == 0).all()
    np.testing.assert_array_equal(codec.dequantize(codes, s, b, 64), x)
