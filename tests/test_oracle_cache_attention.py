"""Pins of the oracle cache state machine and the oracle attention.  CPU only."""
import numpy as np
import pytest

from oracle import attention, bf16, codec, rotation
from oracle.cache import OracleCache, commit_verified_prefix, commit_verified_snapshot
import seeded_inputs as si


@pytest.fixture(scope="module")
def mb():
    return rotation.blocks_bf16(rotation.build_blocks(si.rotation_draws(0, 256)))


def f32(t):
    return t.float().numpy()


# ---------------------------------------------------------------- cache state machine

def test_cache_matches_list_model(mb):
    rng = np.random.default_rng(0)
    B, H = 2, 2
    c = OracleCache(B, H)
    model = [[[] for _ in range(H)] for _ in range(B)]  # rows of (k_words, v_words)
    step = 0
    for _ in range(25):
        if rng.random() < 0.6:
            n = int(rng.integers(1, 300))
            k, v = si.kv_tokens(3, B, H, n, step=step)
            step += 1
            c.append(f32(k), f32(v), mb)
            kw, _, _ = codec.encode_rows(f32(k), mb, 4, 64)
            vw, _, _ = codec.encode_rows(f32(v), mb, 3, 64)
            for b in range(B):
                for h in range(H):
                    model[b][h].extend(zip(kw[b, h], vw[b, h]))
        else:
            n = rng.integers(0, 400, B)
            t = c.trim(n)
            for b in range(B):
                assert t[b] == min(n[b], len(model[b][0]))
                for h in range(H):
                    del model[b][h][len(model[b][h]) - t[b]:]
        assert c.capacity % 256 == 0 and c.capacity >= c.lens.max()
        for b in range(B):
            assert c.lens[b] == len(model[b][0])
            for h in range(H):
                L = int(c.lens[b])
                if L:
                    np.testing.assert_array_equal(c.k[0][b, h, :L], np.array([r[0] for r in model[b][h]]))
                    np.testing.assert_array_equal(c.v[0][b, h, :L], np.array([r[1] for r in model[b][h]]))


def test_growth_steps_and_nbytes(mb):
    c = OracleCache(1, 2)
    assert c.nbytes() == 0
    k, v = si.kv_tokens(1, 1, 2, 300)
    c.append(f32(k), f32(v), mb)
    assert c.capacity == 512  # ceil(300/256)*256
    # per token-head: K 32 words + V 24 words + 4 scales + 4 biases (bf16) each
    assert c.nbytes() == 2 * 512 * (4 * (32 + 24) + 2 * 2 * 4 * 2)
    k, v = si.kv_tokens(1, 1, 2, 212, step=0)
    c.append(f32(k), f32(v), mb)
    assert c.capacity == 512 and c.lens[0] == 512
    k, v = si.kv_tokens(1, 1, 2, 1, step=1)
    c.append(f32(k), f32(v), mb)
    assert c.capacity == 768


def test_trim_then_append_overwrites_exactly_the_trimmed_rows(mb):
    c = OracleCache(1, 1)
    k, v = si.kv_tokens(2, 1, 1, 100)
    c.append(f32(k), f32(v), mb)
    before = c.k[0][0, 0, :90].copy()
    assert c.trim(10)[0] == 10
    k2, v2 = si.kv_tokens(2, 1, 1, 10, step=5)
    c.append(f32(k2), f32(v2), mb)
    np.testing.assert_array_equal(c.k[0][0, 0, :90], before)
    np.testing.assert_array_equal(c.k[0][0, 0, 90:100], codec.encode_rows(f32(k2), mb, 4, 64)[0][0, 0])
    assert c.trim(1000)[0] == 100 and c.lens[0] == 0


def test_commit_verified_prefix(mb):
    c = OracleCache(3, 1)
    k, v = si.kv_tokens(2, 3, 1, 8)
    c.append(f32(k), f32(v), mb)
    t = commit_verified_prefix(c, 4, np.array([4, 0, 2]))
    assert t.tolist() == [0, 4, 2] and c.lens.tolist() == [8, 4, 6]
    with pytest.raises(ValueError):
        commit_verified_prefix(c, 4, np.array([5, 0, 0]))


def _rows(c, b=0, h=0):
    L = int(c.lens[b])
    return c.k[0][b, h, :L].copy(), c.v[0][b, h, :L].copy()


def test_commit_verified_snapshot_branches(mb):
    """The page's four branches against a list model: stepwise verify appends
    one draft token at a time and snapshots after each; committing accepted_len
    leaves exactly the prefix plus `accepted_len` drafts."""
    base_k, base_v = si.kv_tokens(4, 1, 1, 30)
    drafts = [si.kv_tokens(4, 1, 1, 1, step=s) for s in range(4)]

    def verified_cache():
        c = OracleCache(1, 1)
        c.append(f32(base_k), f32(base_v), mb)
        snaps, states = [], []
        for k, v in drafts:  # verify step i appends draft i, then snapshots
            c.append(f32(k), f32(v), mb)
            snaps.append(c.snapshot())
            states.append(_rows(c))
        return c, snaps, states

    # branch 1: every verified token accepted -> True, cache untouched (holds all 4 drafts)
    c, snaps, states = verified_cache()
    assert commit_verified_snapshot(c, snaps, 4, verified_len=4) is True
    assert int(c.lens[0]) == 34 and all((a == b).all() for a, b in zip(_rows(c), states[3]))
    # branch 2: nothing accepted -> False, cache untouched
    c, snaps, states = verified_cache()
    assert commit_verified_snapshot(c, snaps, 0, verified_len=4) is False
    assert int(c.lens[0]) == 34
    # branch 3: more accepted than snapshots taken -> False, cache untouched
    c, snaps, states = verified_cache()
    assert commit_verified_snapshot(c, snaps[:2], 3, verified_len=4) is False
    assert int(c.lens[0]) == 34
    # branch 4: accepted_len in 1..len(snapshots) -> the state after that many drafts
    for acc in (1, 2, 3):
        c, snaps, states = verified_cache()
        assert commit_verified_snapshot(c, snaps, acc, verified_len=4) is True
        assert int(c.lens[0]) == 30 + acc
        k_rows, v_rows = _rows(c)
        want_k = codec.encode_rows(np.concatenate([f32(base_k)] + [f32(d[0]) for d in drafts[:acc]], axis=2),
                                   mb, 4, 64)[0][0, 0]
        np.testing.assert_array_equal(k_rows, want_k)
        np.testing.assert_array_equal(v_rows, states[acc - 1][1])
        # the restored cache does not alias the snapshot: later appends leave it intact
        c.append(f32(drafts[0][0]), f32(drafts[0][1]), mb)
        np.testing.assert_array_equal(snaps[acc - 1][2][0][0, 0, :30 + acc], want_k)
    # without verified_len the first branch never applies: accepted == len(snapshots) restores the last
    c, snaps, states = verified_cache()
    c.trim(10)
    assert commit_verified_snapshot(c, snaps, 4) is True and int(c.lens[0]) == 34


def test_snapshot_does_not_alias(mb):
    c = OracleCache(1, 1)
    k, v = si.kv_tokens(2, 1, 1, 20)
    c.append(f32(k), f32(v), mb)
    snap = c.snapshot()
    ref = c.k[0][0, 0, :20].copy()
    c.trim(5)
    k2, v2 = si.kv_tokens(2, 1, 1, 5, step=9)
    c.append(f32(k2), f32(v2), mb)
    c.restore(snap)
    np.testing.assert_array_equal(c.k[0][0, 0, :20], ref)
    c.trim(20)
    c.append(f32(k2), f32(v2), mb)
    c.restore(snap)  # a second restore of the same snapshot still sees the original
    np.testing.assert_array_equal(c.k[0][0, 0, :20], ref)


def test_tile_and_keep_row(mb):
    c = OracleCache(1, 2)
    k, v = si.kv_tokens(2, 1, 2, 30)
    c.append(f32(k), f32(v), mb)
    ref = c.v[0][0].copy()
    c.tile(3)
    assert c.batch == 3 and c.lens.tolist() == [30, 30, 30]
    for p in range(3):
        np.testing.assert_array_equal(c.v[0][p], ref)
    c.trim(np.array([1, 2, 3]))
    c.keep_row(2)
    assert c.batch == 1 and c.lens.tolist() == [27]


# ---------------------------------------------------------------- attention

def dense_attention_f32(q, k, v, scale, causal_pos=None):
    """Second, independent formulation: float32 matmuls, explicit 0/1 mask, exp-normalise."""
    s = (q.astype(np.float32) * np.float32(scale)) @ k.astype(np.float32).T
    if causal_pos is not None:
        allowed = np.arange(k.shape[0])[None, :] <= causal_pos[:, None]
        s = np.where(allowed, s, np.float32(-1e30))
    s = s - s.max(axis=1, keepdims=True)
    e = np.exp(s).astype(np.float32)
    return (e @ v.astype(np.float32)) / e.sum(axis=1, keepdims=True)


def build(mb, B, H, n, seed=5, outliers=True):
    c = OracleCache(B, H)
    k, v = si.kv_tokens(seed, B, H, n, outliers=outliers)
    c.append(f32(k), f32(v), mb)
    return c


def test_attention_matches_dense_brute_force(mb):
    c = build(mb, 1, 2, 77)
    q = f32(si.queries(5, 1, 16, 3))
    out = attention.attend(q, c, mb, causal=True)
    m = rotation.dense(mb)
    for h in range(16):
        kh, vh = c.dequantized(0, h // 8)
        qr = codec.rotate(q[0, h], mb)
        o = dense_attention_f32(qr, kh, vh, 1 / 16, np.arange(74, 77))
        np.testing.assert_allclose(out[0, h], o.astype(np.float64) @ m.T, atol=1e-5)


def test_single_token_gives_its_value(mb):
    c = build(mb, 1, 1, 1)
    q = f32(si.queries(6, 1, 1, 1))
    out = attention.attend(q, c, mb)
    _, vh = c.dequantized(0, 0)
    np.testing.assert_allclose(out[0, 0, 0], vh[0] @ rotation.dense(mb).T, atol=1e-12)


def test_identical_keys_and_zero_query_give_the_mean(mb):
    c = build(mb, 1, 1, 50)
    c.k[0][0, 0, :50] = c.k[0][0, 0, 0]
    c.k[1][0, 0, :50] = c.k[1][0, 0, 0]
    c.k[2][0, 0, :50] = c.k[2][0, 0, 0]
    q = f32(si.queries(6, 1, 1, 1))
    _, vh = c.dequantized(0, 0)
    want = vh.mean(0) @ rotation.dense(mb).T
    np.testing.assert_allclose(attention.attend(q, c, mb)[0, 0, 0], want, atol=1e-12)
    c2 = build(mb, 1, 1, 50)
    _, vh2 = c2.dequantized(0, 0)
    out = attention.attend(np.zeros((1, 1, 1, 256), np.float32), c2, mb)
    np.testing.assert_allclose(out[0, 0, 0], vh2.mean(0) @ rotation.dense(mb).T, atol=1e-12)


def test_causal_single_query_equals_no_mask(mb):
    c = build(mb, 2, 2, 40)
    q = f32(si.queries(7, 2, 16, 1))
    np.testing.assert_array_equal(attention.attend(q, c, mb, causal=True), attention.attend(q, c, mb))


def test_gqa_head_mapping(mb):
    c = build(mb, 1, 2, 33)
    q = f32(si.queries(8, 1, 16, 1))
    out = attention.attend(q, c, mb)
    for h in (0, 7, 8, 15):
        kh, vh = c.dequantized(0, h // 8)
        o = attention.attend_slice(q[0, h], kh, vh, mb, 1 / 16, False)
        np.testing.assert_allclose(out[0, h], o, atol=1e-12)
        kx, vx = c.dequantized(0, 1 - h // 8)
        assert not np.allclose(o, attention.attend_slice(q[0, h], kx, vx, mb, 1 / 16, False))


def test_stale_rows_are_never_read(mb):
    c = build(mb, 1, 1, 60)
    c.trim(20)
    q = f32(si.queries(9, 1, 1, 1))
    ref = attention.attend(q, c, mb)
    for arr in c.k + c.v:
        if arr.dtype == np.float32:
            arr[0, 0, 40:] = np.nan
        else:
            arr[0, 0, 40:] = 0xFFFFFFFF
    np.testing.assert_array_equal(attention.attend(q, c, mb), ref)


def test_codec_bypass_rotation_cancels(mb):
    # with exact (unquantised) rotated keys/values the rotated attention equals
    # plain attention up to the bf16 rounding of M and of the rotated vectors
    rng = np.random.default_rng(11)
    k = bf16.round_bf16(rng.standard_normal((64, 256)).astype(np.float32))
    v = bf16.round_bf16(rng.standard_normal((64, 256)).astype(np.float32))
    q = bf16.round_bf16(rng.standard_normal((4, 256)).astype(np.float32))
    kr, vr = codec.rotate(k, mb).astype(np.float64), codec.rotate(v, mb).astype(np.float64)
    rot = attention.attend_slice(q, kr, vr, mb, 1 / 16, False)
    plain = dense_attention_f32(q, k, v, 1 / 16)
    np.testing.assert_allclose(rot, plain, atol=3e-2)


# ---------------------------------------------------------------- explicit masks

def dense_masked_f32(q, k, v, scale, keep=None, add=None):
    """Second formulation with an explicit mask: float32, masked scores dropped
    from the normaliser by index (keep) or added (add), exp-normalise."""
    s = (q.astype(np.float32) * np.float32(scale)) @ k.astype(np.float32).T
    if add is not None:
        s = s + add.astype(np.float32)
    out = np.zeros((q.shape[0], v.shape[1]), np.float32)
    for r in range(q.shape[0]):
        idx = np.arange(k.shape[0]) if keep is None else np.nonzero(keep[r])[0]
        if idx.size == 0:  # nothing kept: every score equal, a uniform average
            idx = np.arange(k.shape[0])
            w = np.ones(idx.size, np.float32)
        else:
            w = np.exp(s[r, idx] - s[r, idx].max())
        out[r] = (w @ v[idx].astype(np.float32)) / w.sum()
    return out


def test_masks_match_dense_brute_force(mb):
    c = build(mb, 1, 2, 45)
    q = f32(si.queries(21, 1, 16, 3))
    rng = np.random.default_rng(22)
    keep = rng.random((1, 3, 64)) < 0.6
    keep[0, 1, :] = False  # one row with every key masked
    add = rng.standard_normal((1, 3, 64)).astype(np.float32)
    add[0, 2, ::3] = -np.inf
    out_keep = attention.attend(q, c, mb, mask=keep)
    out_add = attention.attend(q, c, mb, mask=add)
    m = rotation.dense(mb)
    for h in (0, 5, 9, 15):
        kh, vh = c.dequantized(0, h // 8)
        qr = codec.rotate(q[0, h], mb)
        o = dense_masked_f32(qr, kh, vh, 1 / 16, keep=keep[0, :, :45])
        np.testing.assert_allclose(out_keep[0, h], o.astype(np.float64) @ m.T, atol=1e-5)
        o = dense_masked_f32(qr, kh, vh, 1 / 16, add=add[0, :, :45])
        np.testing.assert_allclose(out_add[0, h], o.astype(np.float64) @ m.T, atol=1e-5)


def test_mask_special_cases(mb):
    c = build(mb, 2, 2, 40)
    q = f32(si.queries(23, 2, 16, 4))
    plain = attention.attend(q, c, mb)
    # all-True bool mask, all-zero and constant additive masks: no mask
    np.testing.assert_array_equal(attention.attend(q, c, mb, mask=np.ones((2, 4, 48), bool)), plain)
    np.testing.assert_array_equal(attention.attend(q, c, mb, mask=np.zeros((2, 4, 48), np.float32)), plain)
    np.testing.assert_allclose(attention.attend(q, c, mb, mask=np.full((2, 4, 48), 3.5, np.float32)), plain,
                               atol=1e-12)
    # the causal pattern as a bool mask, and as -inf added: causal
    causal = attention.attend(q, c, mb, causal=True)
    keep = np.arange(48)[None, None, :] <= (40 - 4 + np.arange(4))[None, :, None]
    keep = np.broadcast_to(keep, (2, 4, 48))
    np.testing.assert_array_equal(attention.attend(q, c, mb, mask=keep), causal)
    np.testing.assert_array_equal(attention.attend(q, c, mb, mask=np.where(keep, 0.0, -np.inf)), causal)
    # every key masked: the uniform mean of the values
    none = np.zeros((2, 4, 48), bool)
    out = attention.attend(q, c, mb, mask=none)
    for b in range(2):
        for h in (0, 8):
            _, vh = c.dequantized(b, h // 8)
            np.testing.assert_allclose(out[b, h, 2], vh.mean(0) @ rotation.dense(mb).T, atol=1e-12)
    with pytest.raises(ValueError):
        attention.attend(q, c, mb, causal=True, mask=keep)


# ---------------------------------------------------------------- other formats

FORMATS = [(2, 2, 32), (3, 5, 128), (5, 6, 64), (8, 8, 128), (6, 3, 32)]


@pytest.mark.parametrize("kb,vb,gs", FORMATS)
def test_other_formats_decode_within_the_quantiser_bound(mb, kb, vb, gs):
    """Rows of a cache in another format (widths 2-8, groups 32/64/128) decode
    to the rotated inputs within the quantiser's error bound, after an append,
    a trim and an append over the trimmed rows."""
    c = OracleCache(2, 1, k_bits=kb, v_bits=vb, group_size=gs)
    k1, v1 = si.kv_tokens(40, 2, 1, 50, outliers=True)
    k2, v2 = si.kv_tokens(41, 2, 1, 30, outliers=True)
    c.append(f32(k1), f32(v1), mb)
    c.trim(np.array([20, 0]))
    c.append(f32(k2), f32(v2), mb)
    assert c.lens.tolist() == [60, 80]
    for b in range(2):
        keep = 30 if b == 0 else 50
        for x_all, bits, which in ((np.concatenate([f32(k1)[b, 0, :keep], f32(k2)[b, 0]]), kb, 0),
                                   (np.concatenate([f32(v1)[b, 0, :keep], f32(v2)[b, 0]]), vb, 1)):
            xr = codec.rotate(x_all, mb).astype(np.float64)
            deq = c.dequantized(b, 0)[which]
            assert c.k[0].shape[-1] == 256 * kb // 32 and c.v[0].shape[-1] == 256 * vb // 32
            g = xr.reshape(len(xr), 256 // gs, gs)
            s = (c.k if which == 0 else c.v)[1][b, 0, :len(xr)].astype(np.float64)
            scale = (g.max(-1) - g.min(-1)) / (2 ** bits - 1)
            bound = s / 2 + (2 ** bits - 1) * np.abs(scale - s) + 1e-6 * np.abs(g).max(-1)
            err = np.abs(deq.reshape(g.shape) - g)
            assert (err <= bound[..., None]).all()


@pytest.mark.parametrize("kb,vb,gs", FORMATS)
def test_other_formats_attention_matches_dense_brute_force(mb, kb, vb, gs):
    c = OracleCache(1, 2, k_bits=kb, v_bits=vb, group_size=gs)
    k, v = si.kv_tokens(42, 1, 2, 45, outliers=True)
    c.append(f32(k), f32(v), mb)
    q = f32(si.queries(43, 1, 16, 2))
    out = attention.attend(q, c, mb, causal=True)
    m = rotation.dense(mb)
    for h in range(16):
        kh, vh = c.dequantized(0, h // 8)
        qr = codec.rotate(q[0, h], mb)
        o = dense_attention_f32(qr, kh, vh, 1 / 16, np.arange(43, 45))
        np.testing.assert_allclose(out[0, h], o.astype(np.float64) @ m.T, atol=1e-5)
