"""Rotated K4/V3 bit-packed KV cache and GQA attention for one sm_103a GPU.

The compute lives in `libiqkv.so` (CUDA kernels behind the C ABI declared in
`include/iqkv.h`); this package only marshals arguments.  Importing it does not
load the library; the first call that needs it does, and raises ImportError if
the library has not been built.
"""
from .cache import IQCache, Rotation, commit_verified_snapshot  # noqa: F401
from ._abi import IQError, LIB_PATH  # noqa: F401
