"""CPU oracle for the rotated K4/V3 quantised KV cache — TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously-correct NumPy restatement of what the pages compute:

* page "sparkle mlx_streaming/core/cache/quant_kv.py": `_quat_left`,
  `_quat_right_conj`, `build_block_so4`, `rotate_last`, `_packed_words`,
  `AsymmetricQuantizedKVCache` (`update_and_fetch`, `trim`, `state`) and
  `asym_quantized_sdpa`;
* page "sparkle mlx_streaming/mtp/kv_cache.py": `commit_verified_prefix`
  (trim branch), `_snapshot`/`_restore`, `tile_caches`/`commit_tree_row`.

Only the tests, the smoke check and the benchmark's CPU-baseline / reference
arm may import this package.  The product path (the `libiqkv` C-ABI library and
its Python binding) never imports, calls or links anything here, and nothing
here imports the product.  The oracle shares no code with the CUDA path; the
one shared module is `seeded_inputs`, which draws random numbers only.

Every function here has a pin in `tests/test_oracle_*.py` that checks it
against something other than itself (closed forms, invariants, brute force,
textbook routines, hand-worked fixtures under `tests/golden/`).
"""
from . import bf16, rotation, codec, cache, attention  # noqa: F401
