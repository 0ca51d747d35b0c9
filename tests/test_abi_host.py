"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/bsfp8.h declares, and rejects bad arguments with the
documented codes before touching a device."""
import ctypes
import os
import re

import pytest

import block_scaled_fp8_sm_gb300 as bs
from block_scaled_fp8_sm_gb300 import _abi

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "bsfp8.h")


@pytest.fixture(scope="module")
def lib():
    from block_scaled_fp8_sm_gb300 import build
    build.build()
    return bs.library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8_[a-z_0-9]+)\s*\(", text)))


def test_header_declarations_match_binding():
    assert _declared_functions() == sorted(_abi.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version_and_strerror(lib):
    assert bs.fp8_version() == 10000
    for code in range(0, -10, -1):
        assert bs.fp8_strerror(code).startswith("FP8_")
    assert "unknown" in bs.fp8_strerror(-99)


def _call(lib, A=16, sA=16, B=16, sB=16, C=16, M=64, N=64, K=64, mode=0):
    return lib.fp8_gemm_blockscaled_ex(A, sA, B, sB, C, M, N, K, mode, None)


def test_shape_errors(lib):
    assert _call(lib, N=33) == _abi.FP8_ERR_SHAPE
    assert _call(lib, K=48) == _abi.FP8_ERR_SHAPE
    assert _call(lib, M=-1) == _abi.FP8_ERR_SHAPE
    assert _call(lib, M=1 << 31) == _abi.FP8_ERR_SHAPE
    assert _call(lib, mode=7) == _abi.FP8_ERR_MODE


def test_pertoken_argument_errors(lib):
    def call(mode=0, **kw):
        a = dict(A=16, sA=16, B=16, sB=16, C=16, M=64, N=64, K=64)
        a.update(kw)
        return lib.fp8_gemm_pertoken_ex(a["A"], a["sA"], a["B"], a["sB"], a["C"], a["M"], a["N"], a["K"], mode, None)
    assert call(mode=7) == _abi.FP8_ERR_MODE
    assert call(mode=-1) == _abi.FP8_ERR_MODE
    assert call(N=33, mode=_abi.FP8_PATH_NATIVE) == _abi.FP8_ERR_SHAPE
    assert call(K=48, mode=_abi.FP8_PATH_NATIVE) == _abi.FP8_ERR_SHAPE
    assert call(C=0, mode=_abi.FP8_PATH_NATIVE) == _abi.FP8_ERR_NULL
    assert call(C=8, mode=_abi.FP8_PATH_NATIVE) == _abi.FP8_ERR_ALIGN
    assert call(sA=2, mode=_abi.FP8_PATH_NATIVE) == _abi.FP8_ERR_ALIGN
    assert call(A=0, sA=0, B=0, sB=0, C=0, M=0, mode=_abi.FP8_PATH_NATIVE) == _abi.FP8_OK


def test_quant_out_argument_errors(lib):
    def call(**kw):
        a = dict(A=16, sA=16, B=16, sB=16, Cq=16, sC=16, M=64, N=64, K=64)
        a.update(kw)
        return lib.fp8_gemm_blockscaled_quant(a["A"], a["sA"], a["B"], a["sB"], a["Cq"], a["sC"],
                                              a["M"], a["N"], a["K"], None)
    assert call(N=33) == _abi.FP8_ERR_SHAPE
    assert call(K=48) == _abi.FP8_ERR_SHAPE
    assert call(M=-1) == _abi.FP8_ERR_SHAPE
    assert call(Cq=0) == _abi.FP8_ERR_NULL
    assert call(sC=0) == _abi.FP8_ERR_NULL
    assert call(A=0) == _abi.FP8_ERR_NULL
    assert call(Cq=8) == _abi.FP8_ERR_ALIGN
    assert call(sC=2) == _abi.FP8_ERR_ALIGN
    assert call(B=24) == _abi.FP8_ERR_ALIGN
    assert call(A=0, sA=0, B=0, sB=0, Cq=0, sC=0, M=0) == _abi.FP8_OK


def test_pertoken_e8m0_argument_errors(lib):
    def call(**kw):
        a = dict(A=16, sA=1, B=16, sB=16, C=16, M=64, N=64, K=64)
        a.update(kw)
        return lib.fp8_gemm_pertoken_e8m0(a["A"], a["sA"], a["B"], a["sB"], a["C"], a["M"], a["N"], a["K"], None)
    assert call(N=33) == _abi.FP8_ERR_SHAPE
    assert call(K=48) == _abi.FP8_ERR_SHAPE
    assert call(C=0) == _abi.FP8_ERR_NULL
    assert call(sA=0) == _abi.FP8_ERR_NULL
    assert call(C=8) == _abi.FP8_ERR_ALIGN
    assert call(sB=2) == _abi.FP8_ERR_ALIGN
    assert call(A=0, sA=0, B=0, sB=0, C=0, M=0) == _abi.FP8_OK


def test_empty_problems_enqueue_nothing(lib):
    # M == 0 or N == 0: OK without any device work (no device needed)
    assert _call(lib, A=0, sA=0, B=0, sB=0, C=0, M=0) == _abi.FP8_OK
    assert _call(lib, A=0, sA=0, B=0, sB=0, C=0, N=0) == _abi.FP8_OK
    arr = (_abi.fp8_group_desc * 1)()
    assert lib.fp8_gemm_grouped(arr, 16, 64, 64, 0, None) == _abi.FP8_OK


def test_null_and_alignment_errors(lib):
    assert _call(lib, A=0) == _abi.FP8_ERR_NULL
    assert _call(lib, C=0) == _abi.FP8_ERR_NULL
    assert _call(lib, A=24) == _abi.FP8_ERR_ALIGN
    assert _call(lib, C=8) == _abi.FP8_ERR_ALIGN
    assert _call(lib, sA=18) == _abi.FP8_ERR_ALIGN
    arr = (_abi.fp8_group_desc * 2)()
    arr[0] = _abi.fp8_group_desc(16, 16, 16, 16, 16)
    arr[1] = _abi.fp8_group_desc(16, 16, 0, 16, 16)
    assert lib.fp8_gemm_grouped(arr, 16, 64, 64, 2, None) == _abi.FP8_ERR_NULL
    arr[1] = _abi.fp8_group_desc(16, 16, 40, 16, 16)
    assert lib.fp8_gemm_grouped(arr, 16, 64, 64, 2, None) == _abi.FP8_ERR_ALIGN
    assert lib.fp8_gemm_grouped(arr, 16, 64, 64, -1, None) == _abi.FP8_ERR_SHAPE
    assert lib.fp8_gemm_grouped(arr, 0, 64, 64, 2, None) == _abi.FP8_ERR_NULL


def test_quantize_argument_errors(lib):
    q = lib.fp8_quantize_blocks
    assert q(16, 16, 16, 64, 48, None) == _abi.FP8_ERR_SHAPE       # K not a multiple of 32
    assert q(16, 16, 16, -1, 64, None) == _abi.FP8_ERR_SHAPE
    assert q(16, 16, 16, 1 << 31, 64, None) == _abi.FP8_ERR_SHAPE
    assert q(0, 0, 0, 0, 64, None) == _abi.FP8_OK                   # empty: nothing enqueued
    assert q(0, 16, 16, 64, 64, None) == _abi.FP8_ERR_NULL
    assert q(16, 16, 0, 64, 64, None) == _abi.FP8_ERR_NULL
    assert q(24, 16, 16, 64, 64, None) == _abi.FP8_ERR_ALIGN
    assert q(16, 8, 16, 64, 64, None) == _abi.FP8_ERR_ALIGN
    assert q(16, 16, 18, 64, 64, None) == _abi.FP8_ERR_ALIGN


def test_rowcol_argument_errors(lib):
    r = lib.fp8_gemm_rowcol
    assert r(16, 16, 16, 16, 16, 64, 33, 64, None) == _abi.FP8_ERR_SHAPE
    assert r(16, 16, 16, 16, 16, 64, 64, 48, None) == _abi.FP8_ERR_SHAPE
    assert r(0, 0, 0, 0, 0, 0, 64, 64, None) == _abi.FP8_OK            # M == 0: nothing enqueued
    assert r(16, 0, 16, 16, 16, 64, 64, 64, None) == _abi.FP8_ERR_NULL
    assert r(16, 16, 16, 16, 8, 64, 64, 64, None) == _abi.FP8_ERR_ALIGN
    assert r(16, 18, 16, 16, 16, 64, 64, 64, None) == _abi.FP8_ERR_ALIGN


def test_residual_argument_errors(lib):
    r = lib.fp8_gemm_blockscaled_residual
    assert r(16, 16, 16, 16, 16, 16, 64, 33, 64, None) == _abi.FP8_ERR_SHAPE
    assert r(0, 0, 0, 0, 0, 0, 0, 64, 64, None) == _abi.FP8_OK          # M == 0: nothing enqueued
    assert r(16, 16, 16, 16, 0, 16, 64, 64, 64, None) == _abi.FP8_ERR_NULL
    assert r(16, 16, 16, 16, 8, 16, 64, 64, 64, None) == _abi.FP8_ERR_ALIGN
    assert r(16, 16, 16, 16, 16, 8, 64, 64, 64, None) == _abi.FP8_ERR_ALIGN


def test_debug_keys(lib):
    assert lib.fp8_debug_set(1, 12345) == _abi.FP8_OK
    assert lib.fp8_debug_set(1, 0) == _abi.FP8_OK
    assert lib.fp8_debug_set(2, -1) == _abi.FP8_OK
    assert lib.fp8_debug_set(99, 0) == _abi.FP8_ERR_MODE


def test_binding_raises_on_error(lib):
    class T:
        def __init__(self, p, shape=(64, 64)):
            self.p, self.shape = p, shape

        def data_ptr(self):
            return self.p

    with pytest.raises(bs.Fp8Error) as e:
        bs.fp8_gemm_blockscaled(T(16), T(16), T(16, (33, 64)), T(16), T(16), stream=0)
    assert e.value.code == _abi.FP8_ERR_SHAPE


def test_grouped_device_argument_errors(lib):
    """fp8_gemm_grouped_device checks its host-visible arguments before any
    device work: sizes, null and misaligned pointers, a short workspace."""
    need = lib.fp8_grouped_workspace_bytes(4)
    assert need >= 4 * 128
    assert lib.fp8_grouped_workspace_bytes(-1) == 0
    f = lib.fp8_gemm_grouped_device
    assert f(256, 256, 64, 64, -1, 256, need, None) == _abi.FP8_ERR_SHAPE
    assert f(256, 256, 48, 64, 4, 256, need, None) == _abi.FP8_ERR_SHAPE
    assert f(0, 0, 64, 64, 0, 0, 0, None) == _abi.FP8_OK            # G = 0: nothing to do
    assert f(256, 256, 0, 64, 4, 256, need, None) == _abi.FP8_OK    # N = 0: nothing to do
    assert f(256, 256, 64, 64, 4, 0, need, None) == _abi.FP8_ERR_NULL
    assert f(256, 256, 64, 64, 4, 256 + 64, need, None) == _abi.FP8_ERR_ALIGN
    assert f(256, 256, 64, 64, 4, 256, need - 1, None) == _abi.FP8_ERR_SHAPE
