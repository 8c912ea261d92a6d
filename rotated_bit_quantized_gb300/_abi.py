"""ctypes declarations of libiqkv (include/iqkv.h).  Argument marshalling only.

Loading fails loudly when the shared library has not been built: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libiqkv.so")

IQ_OK = 0
IQ_ERR_INVALID_ARG = 1
IQ_ERR_CAPACITY = 2
IQ_ERR_WORKSPACE = 3
IQ_ERR_UNSUPPORTED = 4
IQ_ERR_CUDA = 5
IQ_ERR_DEVICE = 6
IQ_MAX_BATCH = 256
IQ_STEP = 256
IQ_NOALLOC_SCRATCH_BYTES = 16 << 20
IQ_MASK_NONE, IQ_MASK_CAUSAL, IQ_MASK_ADD_F32, IQ_MASK_BOOL_U8 = 0, 1, 2, 3
IQ_INJECT_COMBINE_WAIT, IQ_INJECT_STAGE_NEVER_FILLED = 1, 2
IQ_DTYPE_BF16, IQ_DTYPE_F32 = 0, 1

EXPORTS = ("iq_status_string", "iq_last_error", "iq_build_rotation", "iq_cache_bytes",
           "iq_cache_check", "iq_cache_nbytes", "iq_cache_append", "iq_cache_trim",
           "iq_cache_gather", "iq_attend_workspace", "iq_attend", "iq_read_status",
           "iq_attend_noalloc", "iq_cache_append_attend", "iq_attend_mask", "iq_noalloc_read_status",
           "iq_debug_inject", "iq_cache_alloc", "iq_cache_grow")


class IQCacheDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("k_bits", ctypes.c_int32), ("v_bits", ctypes.c_int32),
                ("capacity", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("k_codes", ctypes.c_void_p), ("k_scales", ctypes.c_void_p),
                ("k_biases", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("v_scales", ctypes.c_void_p), ("v_biases", ctypes.c_void_p),
                ("lens", ctypes.POINTER(ctypes.c_int32))]


class IQError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str):
        super().__init__(f"{where}: {status_name(code)}: {detail}")
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libiqkv.so is not built ({LIB_PATH}); run __graft_entry__.build() "
                              "or python rotated_bit_quantized_gb300/build.py")
        L = ctypes.CDLL(LIB_PATH)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        DESC = ctypes.POINTER(IQCacheDesc)
        I32P = ctypes.POINTER(ctypes.c_int32)
        L.iq_status_string.argtypes, L.iq_status_string.restype = [I], ctypes.c_char_p
        L.iq_last_error.argtypes, L.iq_last_error.restype = [], ctypes.c_char_p
        L.iq_build_rotation.argtypes = [I, P, P, P, P]
        L.iq_cache_bytes.argtypes = [I, I, I, I, I, I, I, I, ctypes.POINTER(S)]
        L.iq_cache_check.argtypes = [DESC]
        L.iq_cache_nbytes.argtypes, L.iq_cache_nbytes.restype = [DESC], S
        L.iq_cache_append.argtypes = [DESC, P, P, I, P, P]
        L.iq_cache_trim.argtypes = [DESC, I32P, I32P]
        L.iq_cache_gather.argtypes = [DESC, DESC, I32P, P]
        L.iq_attend_workspace.argtypes = [DESC, I, I, ctypes.POINTER(S)]
        L.iq_attend.argtypes = [DESC, P, I, I, ctypes.c_float, I, P, P, I, P, S, P]
        L.iq_read_status.argtypes = [P, P, ctypes.POINTER(I)]
        L.iq_attend_noalloc.argtypes = [DESC, P, I, I, ctypes.c_float, I, P, P, I, P]
        L.iq_cache_append_attend.argtypes = [DESC, P, P, I, P, I, I, ctypes.c_float, I, P, P, I, P, S, P]
        L.iq_attend_mask.argtypes = [DESC, P, I, I, ctypes.c_float, I, P, ctypes.c_longlong, P, P, I, P, S, P]
        L.iq_noalloc_read_status.argtypes = [P, ctypes.POINTER(I)]
        L.iq_debug_inject.argtypes = [I, ctypes.c_uint, ctypes.c_ulonglong]
        L.iq_cache_alloc.argtypes = [DESC, I, I, I, I, I, I, I, I, ctypes.POINTER(P), I32P]
        L.iq_cache_grow.argtypes = [DESC, DESC, P]
        for name in EXPORTS:
            if name not in ("iq_status_string", "iq_last_error", "iq_cache_nbytes"):
                getattr(L, name).restype = I
        _lib = L
    return _lib


def status_name(code: int) -> str:
    return lib().iq_status_string(code).decode()


def check(code: int, where: str) -> None:
    if code != IQ_OK:
        raise IQError(code, where, lib().iq_last_error().decode())
