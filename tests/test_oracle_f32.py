"""Pins of the oracle's float32 path (float32 keys, values and queries, float32
scales and biases, the float32 rotation blocks) against things other than
itself: hand-worked fixtures (tests/golden/float32_inputs.json), the float32
error bound of a 4-term dot product against float64, closed forms of the
quantiser and a dense brute-force attention.  CPU only."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import attention, bf16, codec, rotation
from oracle.cache import OracleCache
import seeded_inputs as si

GOLD = os.path.join(os.path.dirname(__file__), "golden")
U = 2.0 ** -24  # float32 unit roundoff


@pytest.fixture(scope="module")
def gold():
    with open(os.path.join(GOLD, "float32_inputs.json")) as f:
        return json.load(f)


@pytest.fixture(scope="module")
def m32():
    return rotation.build_blocks(si.rotation_draws(0, 256))


def f32(t):
    return t.float().numpy()


def identity_blocks():
    return np.tile(np.eye(4, dtype=np.float32), (64, 1, 1))


# ---------------------------------------------------------------- rotation

def test_golden_rotate_order(gold):
    g = gold["rotate_order"]
    blocks = identity_blocks()
    blocks[0] = 1.0
    x = np.zeros(256, np.float32)
    x[:4] = g["x_head"]
    y = codec.rotate_f32(x[None], blocks)[0]
    assert y[:4].tolist() == g["y_head"], g["derivation"]
    assert not y[4:].any()


def test_golden_rotate_rounds_each_product(gold):
    g = gold["rotate_separate_rounding"]
    blocks = identity_blocks()
    blocks[0] = 0.0
    blocks[0, :, 0] = g["m_col0"]
    x = np.zeros(256, np.float32)
    x[:4] = g["x_head"]
    y = codec.rotate_f32(x[None], blocks)[0]
    assert y[:4].tolist() == g["y_head"], g["derivation"]


def test_rotate_f32_unit_vectors_give_rows_of_m(m32):
    """e_i @ M is row i of M exactly (one product by 1, sums with zeros)."""
    dense = rotation.dense(m32)
    for i in (0, 1, 2, 3, 77, 255):
        e = np.zeros((1, 256), np.float32)
        e[0, i] = 1.0
        np.testing.assert_array_equal(codec.rotate_f32(e, m32)[0], dense[i].astype(np.float32))


def test_rotate_f32_within_float32_dot_product_bound(m32):
    """|fl(x @ M) - x @ M| <= gamma_4 * sum |x_i M_ij| (four products and three
    sums, each one rounding), against the exact product in float64; a
    transposed block or a dropped term would break it."""
    rng = np.random.default_rng(81)
    x = (rng.standard_normal((200, 256)) * rng.uniform(0.01, 50, (200, 1))).astype(np.float32)
    got = codec.rotate_f32(x, m32).astype(np.float64)
    dense = rotation.dense(m32).astype(np.float64)
    exact = x.astype(np.float64) @ dense
    gamma4 = 4 * U / (1 - 4 * U)
    bound = gamma4 * (np.abs(x.astype(np.float64)) @ np.abs(dense))
    assert (np.abs(got - exact) <= bound).all()
    assert not np.allclose(got, x.astype(np.float64) @ dense.T, atol=1e-3)


def test_rotate_f32_keeps_float32_precision(m32):
    """Unlike the bfloat16 path nothing is rounded to bfloat16: the outputs are
    mostly not bfloat16 values, and they preserve norms to float32 accuracy."""
    rng = np.random.default_rng(82)
    x = rng.standard_normal((50, 256)).astype(np.float32)
    y = codec.rotate_f32(x, m32)
    assert np.mean(bf16.round_bf16(y) == y) < 0.05
    np.testing.assert_allclose(np.linalg.norm(y.astype(np.float64), axis=1),
                               np.linalg.norm(x.astype(np.float64), axis=1), rtol=1e-5)


# ---------------------------------------------------------------- quantiser

def test_golden_quantize_f32_exact(gold):
    g = gold["quantize_f32_exact"]
    k = np.array(g["k"], np.float64)
    x = (np.float64(g["b"]) + k * np.float64(g["s"])).astype(np.float32)
    assert np.array_equal(x.astype(np.float64), g["b"] + k * g["s"])  # every input exact in float32
    codes, s, b = codec.quantize(x[None], g["bits"], g["group_size"], meta="f32")
    assert s[0, 0] == np.float32(g["s_hat_f32"]) and b[0, 0] == np.float32(g["b"]), g["derivation"]
    assert codes[0].tolist() == g["k"]
    np.testing.assert_array_equal(codec.dequantize(codes, s, b, g["group_size"])[0], x.astype(np.float64))
    _, s_b, _ = codec.quantize(x[None], g["bits"], g["group_size"], meta="bf16")
    assert s_b[0, 0] == np.float32(g["s_hat_bf16"])


@pytest.mark.parametrize("gs", [32, 64, 128])
@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_quantize_f32_bound_and_extremes(bits, gs):
    """float32 scale kept as computed: |x - deq| <= s/2 (plus float32 rounding
    of the difference and the quotient), the minimum codes to 0 and the
    maximum to exactly 2^b - 1."""
    rng = np.random.default_rng(90 + bits + gs)
    x = (rng.standard_normal((400, 256)) * rng.uniform(0.1, 30, (400, 1))).astype(np.float32)
    codes, s, b = codec.quantize(x, bits, gs, meta="f32")
    g = x.reshape(400, 256 // gs, gs).astype(np.float64)
    scale = (g.max(-1) - g.min(-1)) / (2 ** bits - 1)
    np.testing.assert_allclose(s, scale, rtol=2 * U)  # one rounding of the difference, one of the quotient
    deq = codec.dequantize(codes, s, b, gs).reshape(g.shape)
    bound = s.astype(np.float64) / 2 * (1 + 1e-5) + 4 * U * np.abs(g).max(-1)
    assert (np.abs(deq - g) <= bound[..., None]).all()
    cg = codes.reshape(g.shape)
    assert (np.take_along_axis(cg, g.argmin(-1)[..., None], -1) == 0).all()
    assert (np.take_along_axis(cg, g.argmax(-1)[..., None], -1) == 2 ** bits - 1).all()


def test_quantize_f32_brute_force_nearest_level():
    rng = np.random.default_rng(95)
    x = rng.standard_normal((300, 64)).astype(np.float32)
    for bits in (2, 3, 4, 5, 6, 8):
        codes, s, b = codec.quantize(x, bits, 64, meta="f32")
        levels = s[:, :, None].astype(np.float64) * np.arange(2 ** bits) + b[:, :, None]
        dist = np.abs(x.astype(np.float64)[:, :, None] - levels[:, 0][:, None, :])
        mine = np.take_along_axis(dist, codes.astype(int)[..., None], -1)[..., 0]
        assert np.all(mine - dist.min(-1) <= 1e-6 * (1 + np.abs(x)))


# ---------------------------------------------------------------- cache and attention

def test_f32_cache_stores_float32_metadata(m32):
    """Scales are the float32 scales of the float32 rotated rows (mostly not
    bfloat16 values) and nbytes counts 4 bytes per scale and bias."""
    c = OracleCache(1, 2, dtype="f32")
    k, v = si.kv_tokens(61, 1, 2, 40, outliers=True, dtype=torch.float32)
    c.append(f32(k), f32(v), m32)
    xr = codec.rotate_f32(f32(k)[0, 1], m32).reshape(40, 4, 64).astype(np.float64)
    want = ((xr.max(-1) - xr.min(-1)).astype(np.float32) / np.float32(15)).astype(np.float32)
    np.testing.assert_array_equal(c.k[1][0, 1, :40], want)
    np.testing.assert_array_equal(c.k[2][0, 1, :40], xr.min(-1).astype(np.float32))
    assert np.mean(bf16.round_bf16(c.k[1][0, 1, :40]) == c.k[1][0, 1, :40]) < 0.1
    assert c.nbytes() == 1 * 2 * 256 * (4 * (32 + 24) + 4 * 4 * 4)


def dense_attention_f64(q, k, v, scale, causal_pos=None):
    """Independent formulation: explicit 0/1 mask, exp-normalise, float64."""
    s = (q.astype(np.float64) * scale) @ k.T
    if causal_pos is not None:
        allowed = np.arange(k.shape[0])[None, :] <= causal_pos[:, None]
        s = np.where(allowed, s, -1e300)
    e = np.exp(s - s.max(axis=1, keepdims=True))
    return (e @ v) / e.sum(axis=1, keepdims=True)


def test_f32_attention_matches_dense_brute_force(m32):
    c = OracleCache(1, 2, dtype="f32")
    k, v = si.kv_tokens(62, 1, 2, 70, outliers=True, dtype=torch.float32)
    c.append(f32(k), f32(v), m32)
    q = f32(si.queries(63, 1, 16, 3, dtype=torch.float32))
    out = attention.attend(q, c, m32, causal=True)
    dense = rotation.dense(m32).astype(np.float64)
    for h in range(16):
        kh, vh = c.dequantized(0, h // 8)
        qr = codec.rotate_f32(q[0, h], m32)
        o = dense_attention_f64(qr, kh, vh, 1 / 16, np.arange(67, 70))
        np.testing.assert_allclose(out[0, h], o @ dense.T, atol=1e-9)


def test_f32_single_token_and_decode_close_to_unquantised(m32):
    """T = 1 returns the token's dequantised value rotated back; with 8-bit
    codes the float32 cache's attention is close to exact attention over the
    unquantised float32 inputs (the rotation cancels)."""
    c = OracleCache(1, 1, dtype="f32")
    k, v = si.kv_tokens(64, 1, 1, 1, dtype=torch.float32)
    c.append(f32(k), f32(v), m32)
    q = f32(si.queries(65, 1, 1, 1, dtype=torch.float32))
    _, vh = c.dequantized(0, 0)
    dense = rotation.dense(m32).astype(np.float64)
    np.testing.assert_allclose(attention.attend(q, c, m32)[0, 0, 0], vh[0] @ dense.T, atol=1e-12)
    c8 = OracleCache(1, 1, k_bits=8, v_bits=8, dtype="f32")
    k, v = si.kv_tokens(66, 1, 1, 300, dtype=torch.float32)
    c8.append(f32(k), f32(v), m32)
    q = f32(si.queries(67, 1, 1, 1, dtype=torch.float32))
    exact = dense_attention_f64(q[0, 0].astype(np.float64), f32(k)[0, 0].astype(np.float64),
                                f32(v)[0, 0].astype(np.float64), 1 / 16)
    np.testing.assert_allclose(attention.attend(q, c8, m32)[0, 0], exact, atol=2e-2)
