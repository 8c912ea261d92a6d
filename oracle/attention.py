"""GQA attention over the quantised cache (oracle side).

Page "sparkle mlx_streaming/core/cache/quant_kv.py", `asym_quantized_sdpa`:
queries are scaled, reshaped so that query head h reads kv head h // rep
(rep = Hq / Hkv), scored against the dequantised keys, masked (a string mask
means causal with query i at absolute position kL - qL + i), soft-maxed, and
multiplied by the dequantised values.  The result is still in rotated value
space; the caller applies the inverse rotation, here `o @ M_b^T`.

Readings:

* The queries are rotated like the keys: q' = bf16(q @ M_b) (same rule as
  `codec.rotate`), then multiplied by the caller's scale (1/sqrt(D)) with the
  product rounded to bfloat16, since the page scales bfloat16 queries
  (`queries * scale`).  For D = 256 the scale is 1/16 and the product is exact.
* Scores, softmax, P*V and the inverse rotation are carried out in float64 on
  the exactly dequantised cache; only the final output is rounded (to
  bfloat16).  The page's MLX kernels would round intermediates to the query
  dtype; the method's accuracy target (bf16 I/O, fp32 accumulation) is read as
  "no intermediate rounding".
* float32 caches (page: `rotate_last` in the queries' dtype, scores in it):
  q' = q @ M with `codec.rotate_f32`, times the scale rounded to float32; the
  inverse rotation uses the float32 blocks of M; a bool mask's masked scores
  become float32's most negative finite value.
* Causally masked scores are -inf (the page uses the dtype's most negative
  finite value; with at least one unmasked key per row the two give the same
  softmax).
* Explicit masks (page: a bool mask selects `where(mask, scores, finfo.min)`,
  a float mask is added to the scores) are read per sequence and query,
  shared by every head: mask [B, L, S] with S >= the sequence length.  A bool
  mask's masked scores become bfloat16's most negative finite value, so a row
  with every key masked averages all values uniformly, as the page's softmax
  would; an additive mask may hold -inf, and a row that is -inf everywhere
  gives NaN, as the page's softmax would.
"""
from __future__ import annotations

import numpy as np

from . import codec
from .bf16 import round_bf16


def inverse_rotate(o, blocks) -> np.ndarray:
    """o @ M^T per 4-wide block in float64 (M_b, or the float32 M of a float32 cache)."""
    o = np.asarray(o, dtype=np.float64)
    m = np.asarray(blocks, dtype=np.float64)
    nb = m.shape[0]
    o4 = o.reshape(o.shape[:-1] + (nb, 4))
    out = np.einsum('...bj,bij->...bi', o4, m)
    return out.reshape(o.shape)


def softmax_rows(s) -> np.ndarray:
    s = np.asarray(s, dtype=np.float64)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=-1, keepdims=True)


BF16_MIN = -3.3895313892515355e38  # most negative finite bfloat16: (2 - 2^-7) * 2^127
F32_MIN = -3.4028234663852886e38   # most negative finite float32: (2 - 2^-23) * 2^127


def attend_slice(q_rows, k_hat, v_hat, blocks, scale, causal, q_pos=None, mask_rows=None, dtype="bf16"):
    """Attention for query rows of one kv head.

    q_rows float32 [R, D] (unrotated; bfloat16 values when dtype is "bf16");
    k_hat, v_hat float64 [T, D]; blocks: M_b ("bf16") or the float32 M ("f32");
    q_pos int [R]: absolute position of each row's query (causal limit t <= q_pos);
    mask_rows [R, T] bool (keep where True) or float (added to the scores).
    Returns float64 [R, D] in unrotated space.
    """
    if dtype == "bf16":
        qr = codec.rotate(q_rows, blocks) * np.float32(scale)
        qr = round_bf16(qr.astype(np.float32)).astype(np.float64)
    else:
        qr = (codec.rotate_f32(q_rows, blocks) * np.float32(scale)).astype(np.float32).astype(np.float64)
    s = qr @ k_hat.T
    if causal:
        t = np.arange(k_hat.shape[0])
        s = np.where(t[None, :] <= np.asarray(q_pos)[:, None], s, -np.inf)
    if mask_rows is not None:
        mask_rows = np.asarray(mask_rows)
        if mask_rows.dtype == np.bool_:
            s = np.where(mask_rows, s, BF16_MIN if dtype == "bf16" else F32_MIN)
        else:
            s = s + mask_rows.astype(np.float64)
    p = softmax_rows(s)
    return inverse_rotate(p @ v_hat, blocks)


def attend(q, cache, blocks, scale=None, causal=False, heads=None, batches=None,
           query_index=None, mask=None):
    """Full oracle attention.

    q float32 [B, Hq, L, D]; blocks: M_b for a "bf16" cache, the float32 M
    for an "f32" one; cache an `OracleCache` already holding the queries'
    own keys/values when causal; mask None or [B, L, S] (bool: keep where True;
    float: added to the scores), S >= every length, shared by the heads.
    Returns float64 [B, Hq, L, D] (entries of skipped rows left as NaN when
    `heads` / `batches` / `query_index` subsample).
    """
    if mask is not None and causal:
        raise ValueError("give either causal or an explicit mask")
    q = np.asarray(q, dtype=np.float32)
    B, Hq, L, D = q.shape
    rep = Hq // cache.kv_heads
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.full(q.shape, np.nan, dtype=np.float64)
    bs = range(B) if batches is None else batches
    hs = range(Hq) if heads is None else heads
    qi = np.arange(L) if query_index is None else np.asarray(query_index)
    for b in bs:
        T = int(cache.lens[b])
        if T <= 0:
            raise ValueError("attention over an empty sequence")
        by_kv = {}
        for h in hs:
            by_kv.setdefault(h // rep, []).append(h)
        for kvh, hl in by_kv.items():
            kh, vh = cache.dequantized(b, kvh)
            rows = q[b, hl][:, qi].reshape(-1, D)
            pos = np.tile(T - L + qi, len(hl))
            mrows = None if mask is None else np.tile(np.asarray(mask[b])[qi, :T], (len(hl), 1))
            o = attend_slice(rows, kh, vh, blocks, scale, causal, pos, mrows, cache.dtype)
            o = o.reshape(len(hl), len(qi), D)
            for j, h in enumerate(hl):
                out[b, h, qi] = o[j]
    return out


def to_bf16(out64) -> np.ndarray:
    """Final output rounding to bfloat16 (via float32), as float32 values."""
    return round_bf16(np.asarray(out64, dtype=np.float32))
