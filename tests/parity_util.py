"""Helpers shared by the GPU parity tests: build matching oracle / device caches
from the seeded inputs and compare results.  Imports the oracle (tests only)."""
from __future__ import annotations

import numpy as np
import torch

import seeded_inputs as si
from oracle import attention, bf16, codec, rotation
from oracle.cache import OracleCache

ATOL = 2e-3  # attention max-abs bound (bf16 I/O, fp32 accumulation)


def oracle_blocks(seed=0):
    return rotation.blocks_bf16(rotation.build_blocks(si.rotation_draws(seed, 256)))


def f32(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy()


def cache_arrays(cache, b, h, n):
    """Device cache rows [0, n) of slice (b, h) as numpy (words uint32, scales/biases f32)."""
    kw = cache.k_codes[b, h, :n].cpu().numpy().view(np.uint32)
    vw = cache.v_codes[b, h, :n].cpu().numpy().view(np.uint32)
    ks = cache.k_scales[b, h, :n].float().cpu().numpy()
    kb = cache.k_biases[b, h, :n].float().cpu().numpy()
    vs = cache.v_scales[b, h, :n].float().cpu().numpy()
    vb = cache.v_biases[b, h, :n].float().cpu().numpy()
    return kw, ks, kb, vw, vs, vb


def assert_rows_equal(cache, b, h, lo, hi, k_rows, v_rows, mb):
    """Device rows [lo, hi) of (b, h) equal the oracle encoding of k_rows / v_rows (bit-exact)."""
    kw, ks, kb = codec.encode_rows(k_rows, mb, 4, 64)
    vw, vs, vb = codec.encode_rows(v_rows, mb, 3, 64)
    got = cache_arrays(cache, b, h, hi)
    want = (kw, ks, kb, vw, vs, vb)
    names = ("k_codes", "k_scales", "k_biases", "v_codes", "v_scales", "v_biases")
    for name, g, w in zip(names, got, want):
        g = g[lo:hi]
        if g.dtype == np.uint32:
            bad = np.count_nonzero(g != w)
            assert bad == 0, f"{name} ({b},{h}) rows {lo}:{hi}: {bad} words differ"
        else:
            np.testing.assert_array_equal(g, w, err_msg=f"{name} ({b},{h}) rows {lo}:{hi}")


def compare_out(out: torch.Tensor, ref64: np.ndarray, what: str, atol: float = ATOL):
    """GPU output vs the oracle's unrounded output on the entries the oracle computed."""
    got = out.float().cpu().numpy()
    mask = ~np.isnan(ref64)
    assert mask.any()
    err = np.abs(got[mask] - ref64[mask])
    if out.dtype == torch.bfloat16:
        bound = atol + 0.5 * bf16.ulp_bf16(ref64[mask])  # bf16 output rounding on top
    else:
        bound = np.full(err.shape, atol)
    worst = float((err - bound).max())
    assert worst <= 0, f"{what}: max abs err {err.max():.3e} exceeds bound by {worst:.3e}"
    assert np.isfinite(got[mask]).all()
    return float(err.max())
