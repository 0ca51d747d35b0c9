"""ctypes declarations of libbsfp8.so (the C ABI in include/bsfp8.h).

Loading never falls back to anything: if the shared library is missing the
import fails with a clear error.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbsfp8.so")

FP8_OK = 0
FP8_ERR_NULL = -1
FP8_ERR_SHAPE = -2
FP8_ERR_ALIGN = -3
FP8_ERR_ARCH = -4
FP8_ERR_CUDA = -5
FP8_ERR_MODE = -6
FP8_ERR_SCALE = -7
FP8_ERR_TIMEOUT = -8
FP8_ERR_RECORD = -9

FP8_PATH_AUTO = 0
FP8_PATH_NATIVE = 1
FP8_PATH_PROMOTE = 2

FP8_DEBUG_WAIT_LIMIT_CYCLES = 1
FP8_DEBUG_WITHHOLD_STAGE = 2
FP8_DEBUG_TRACE_BUFFER = 3

FP8_MAX_GROUPS_PER_LAUNCH = 64

# every symbol include/bsfp8.h declares
EXPORTS = (
    "fp8_gemm_blockscaled", "fp8_gemm_blockscaled_ex", "fp8_gemm_grouped",
    "fp8_gemm_grouped_ex", "fp8_status_query", "fp8_strerror", "fp8_version",
    "fp8_debug_set", "fp8_lib_shutdown", "fp8_gemm_blockscaled_noalloc",
    "fp8_quantize_blocks", "fp8_gemm_rowcol", "fp8_gemm_blockscaled_residual",
    "fp8_gemm_grouped_device", "fp8_grouped_workspace_bytes", "fp8_gemm_pertoken", "fp8_gemm_pertoken_ex",
    "fp8_gemm_blockscaled_quant", "fp8_gemm_pertoken_e8m0",
)


class fp8_group_desc(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("sA", ctypes.c_void_p), ("B", ctypes.c_void_p),
                ("sB", ctypes.c_void_p), ("C", ctypes.c_void_p)]


_lib = None


def load(path: str = None) -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    path = LIB_PATH if path is None else path
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -m block_scaled_fp8_sm_gb300.build` "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    vp, i64, i32, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
    lib.fp8_gemm_blockscaled.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, vp]
    lib.fp8_gemm_blockscaled.restype = ci
    lib.fp8_gemm_blockscaled_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ci, vp]
    lib.fp8_gemm_blockscaled_ex.restype = ci
    lib.fp8_gemm_blockscaled_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, vp]
    lib.fp8_gemm_blockscaled_noalloc.restype = ci
    lib.fp8_quantize_blocks.argtypes = [vp, vp, vp, i64, i64, vp]
    lib.fp8_quantize_blocks.restype = ci
    lib.fp8_gemm_pertoken.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, vp]
    lib.fp8_gemm_pertoken.restype = ci
    lib.fp8_gemm_pertoken_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ci, vp]
    lib.fp8_gemm_pertoken_ex.restype = ci
    lib.fp8_gemm_rowcol.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, vp]
    lib.fp8_gemm_rowcol.restype = ci
    lib.fp8_gemm_blockscaled_residual.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, vp]
    lib.fp8_gemm_blockscaled_residual.restype = ci
    lib.fp8_gemm_blockscaled_quant.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, vp]
    lib.fp8_gemm_blockscaled_quant.restype = ci
    lib.fp8_gemm_pertoken_e8m0.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, vp]
    lib.fp8_gemm_pertoken_e8m0.restype = ci
    lib.fp8_gemm_grouped.argtypes = [ctypes.POINTER(fp8_group_desc), vp, i64, i64, i32, vp]
    lib.fp8_gemm_grouped.restype = ci
    lib.fp8_gemm_grouped_ex.argtypes = [ctypes.POINTER(fp8_group_desc), vp, i64, i64, i32, ci, vp]
    lib.fp8_gemm_grouped_ex.restype = ci
    lib.fp8_gemm_grouped_device.argtypes = [vp, vp, i64, i64, i32, vp, i64, vp]
    lib.fp8_gemm_grouped_device.restype = ci
    lib.fp8_grouped_workspace_bytes.argtypes = [i32]
    lib.fp8_grouped_workspace_bytes.restype = i64
    lib.fp8_status_query.argtypes = [vp, ctypes.POINTER(ci)]
    lib.fp8_status_query.restype = ci
    lib.fp8_strerror.argtypes = [ci]
    lib.fp8_strerror.restype = ctypes.c_char_p
    lib.fp8_version.argtypes = []
    lib.fp8_version.restype = ci
    lib.fp8_debug_set.argtypes = [ci, i64]
    lib.fp8_debug_set.restype = ci
    lib.fp8_lib_shutdown.argtypes = []
    lib.fp8_lib_shutdown.restype = None
    _lib = lib
    return lib
