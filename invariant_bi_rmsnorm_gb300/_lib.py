"""ctypes declarations of libbi.so (the C ABI in include/bi.h).

Loading fails loudly when the library has not been built: there is no
fallback implementation of any kernel.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libbi.so")

# bi_status values (include/bi.h)
BI_OK = 0
BI_ERR_INVALID_ARG = 1
BI_ERR_UNSUPPORTED_SHAPE = 2
BI_ERR_MISALIGNED = 3
BI_ERR_WORKSPACE_TOO_SMALL = 4
BI_ERR_CUDA = 5
BI_ERR_DEVICE_TIMEOUT = 6
BI_ERR_DEVICE_BAD_INPUT = 7

PAGE_SIZE = 16
DECODE_CHUNK = 256
DECODE_COUNTER_BYTES = 262144  # arrival counters at the start of an attention workspace

# every entry point include/bi.h declares
EXPORTS = (
    "bi_abi_version", "bi_status_string", "bi_get_device_error", "bi_rmsnorm", "bi_gemm",
    "bi_decode_attention_workspace_size", "bi_decode_num_chunks", "bi_decode_chunk_len",
    "bi_decode_attention", "bi_decode_attention_noalloc", "bi_decode_attention_fixed_splits",
    "bi_selftest_wait_timeout", "bi_prefill_attention", "bi_prefill_attention_workspace_size",
    "bi_selftest_tcgen05_vs_mma_sync",
    "bi_add_rmsnorm",
    "bi_qk_norm_rope_append", "bi_silu_mul", "bi_decode_attention_launches", "bi_logprobs",
    "bi_gemm_swiglu",
)

_lib = None

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64


def load() -> ctypes.CDLL:
    """Load libbi.so once; raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is not built; run `python -c \"import __graft_entry__ as g; g.build()\"` "
            "(or `python -m invariant_bi_rmsnorm_gb300.build`) first")
    lib = ctypes.CDLL(LIB_PATH)
    lib.bi_abi_version.argtypes = []
    lib.bi_abi_version.restype = ctypes.c_int
    lib.bi_status_string.argtypes = [ctypes.c_int]
    lib.bi_status_string.restype = ctypes.c_char_p
    lib.bi_get_device_error.argtypes = [_vp]
    lib.bi_get_device_error.restype = ctypes.c_int
    lib.bi_rmsnorm.argtypes = [_vp, _vp, _vp, _i64, _i32, _i64, _i64, ctypes.c_float, _vp]
    lib.bi_rmsnorm.restype = ctypes.c_int
    lib.bi_gemm.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _i64, _i64, _i64, _vp]
    lib.bi_gemm.restype = ctypes.c_int
    lib.bi_gemm_swiglu.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _i64, _i64, _i64, _vp]
    lib.bi_gemm_swiglu.restype = ctypes.c_int
    lib.bi_decode_attention_workspace_size.argtypes = [_i32, _i32, _i32, _i32]
    lib.bi_decode_attention_workspace_size.restype = ctypes.c_size_t
    lib.bi_decode_num_chunks.argtypes = [_i32]
    lib.bi_decode_num_chunks.restype = _i32
    lib.bi_decode_chunk_len.argtypes = [_i32, _i32]
    lib.bi_decode_chunk_len.restype = _i32
    lib.bi_decode_attention.argtypes = [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                        _i32, _i32, _i32, ctypes.c_float, _vp, _vp,
                                        ctypes.c_size_t, _vp]
    lib.bi_decode_attention.restype = ctypes.c_int
    lib.bi_decode_attention_noalloc.argtypes = [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32,
                                                _i32, _i32, _i32, _i32, ctypes.c_float, _vp, _vp]
    lib.bi_decode_attention_noalloc.restype = ctypes.c_int
    lib.bi_decode_attention_fixed_splits.argtypes = [
        _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_float,
        _i32, _vp, _vp, ctypes.c_size_t, _vp]
    lib.bi_decode_attention_fixed_splits.restype = ctypes.c_int
    lib.bi_prefill_attention.argtypes = [_vp, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32,
                                         _i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_float, _vp,
                                         _vp, ctypes.c_size_t, _vp]
    lib.bi_prefill_attention.restype = ctypes.c_int
    lib.bi_selftest_tcgen05_vs_mma_sync.argtypes = [_vp] * 10
    lib.bi_selftest_tcgen05_vs_mma_sync.restype = ctypes.c_int
    lib.bi_prefill_attention_workspace_size.argtypes = [_i32, _i32, _i32, _i32]
    lib.bi_prefill_attention_workspace_size.restype = ctypes.c_size_t
    lib.bi_add_rmsnorm.argtypes = [_vp, _vp, _vp, _vp, _i64, _i32, _i64, _i64, _i64,
                                   ctypes.c_float, _vp]
    lib.bi_add_rmsnorm.restype = ctypes.c_int
    lib.bi_qk_norm_rope_append.argtypes = [_vp, _i64, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _i32,
                                           _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _i32, _i32,
                                           _vp]
    lib.bi_qk_norm_rope_append.restype = ctypes.c_int
    lib.bi_silu_mul.argtypes = [_vp, _i64, _i32, _i32, _vp, _i64, _vp]
    lib.bi_silu_mul.restype = ctypes.c_int
    lib.bi_decode_attention_launches.argtypes = [_i32, _i32, _i32]
    lib.bi_decode_attention_launches.restype = _i32
    lib.bi_logprobs.argtypes = [_vp, _i64, _i32, _i64, _vp, _vp, _vp, _vp]
    lib.bi_logprobs.restype = ctypes.c_int
    lib.bi_selftest_wait_timeout.argtypes = [_i32, _vp]
    lib.bi_selftest_wait_timeout.restype = ctypes.c_int
    _lib = lib
    return lib
