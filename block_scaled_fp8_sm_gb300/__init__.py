"""Python binding of libbsfp8 (block-scaled E4M3 GEMM, bf16 out, sm_103a).

Argument marshalling only: torch tensors are turned into device pointers and
the current CUDA stream, and the C entry points of include/bsfp8.h are called
by the same names.  Every step of the computation runs in the library's CUDA
kernels; there is no CPU or library fallback, and a non-zero status raises
``Fp8Error``.
"""
from __future__ import annotations

import ctypes

from . import _abi
from ._abi import (FP8_PATH_AUTO, FP8_PATH_NATIVE, FP8_PATH_PROMOTE,  # noqa: F401
                   FP8_DEBUG_WAIT_LIMIT_CYCLES, FP8_DEBUG_WITHHOLD_STAGE, FP8_DEBUG_TRACE_BUFFER,
                   FP8_MAX_GROUPS_PER_LAUNCH, fp8_group_desc)

__all__ = ["fp8_gemm_blockscaled", "fp8_gemm_blockscaled_noalloc", "fp8_gemm_grouped", "group_descs",
           "fp8_gemm_grouped_device", "fp8_grouped_workspace_bytes", "group_table", "fp8_gemm_pertoken",
           "fp8_quantize_blocks", "fp8_gemm_rowcol", "fp8_gemm_blockscaled_residual",
           "fp8_gemm_blockscaled_quant", "fp8_gemm_pertoken_e8m0", "fp8_status_query", "fp8_strerror", "fp8_version", "fp8_debug_set", "fp8_lib_shutdown",
           "Fp8Error", "library"]


class Fp8Error(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {fp8_strerror(code)} ({code})" if what else fp8_strerror(code))


def library():
    return _abi.load()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check(rc: int, what: str):
    if rc != 0:
        raise Fp8Error(rc, what)


def fp8_gemm_blockscaled(A, sA, B, sB, C, M=None, N=None, K=None, stream=None, mode=None):
    """C[M,N] (bf16) = block-scaled E4M3 GEMM of A[M,K] and B[N,K] with fp32
    32x32 block scales sA, sB.  Tensors are CUDA tensors (A/B uint8 codes or
    float8_e4m3fn, sA/sB float32, C bfloat16).  ``mode`` None = AUTO."""
    M = A.shape[0] if M is None else M
    K = A.shape[1] if K is None else K
    N = B.shape[0] if N is None else N
    lib = library()
    s = _stream(stream)
    if mode is None:
        rc = lib.fp8_gemm_blockscaled(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(C), M, N, K, s)
    else:
        rc = lib.fp8_gemm_blockscaled_ex(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(C), M, N, K,
                                         int(mode), s)
    _check(rc, "fp8_gemm_blockscaled")
    return C


def fp8_gemm_blockscaled_noalloc(A, sA, B, sB, C, M=None, N=None, K=None, stream=None):
    """Same as fp8_gemm_blockscaled (AUTO path) through the entry point that
    allocates no device memory (its status word is a static array inside the
    library).  For callers that cannot allocate device memory, e.g. a server
    whose caching allocator owns the device.  Make the first call on a device
    outside stream capture: it performs that device's one-time set-up."""
    M = A.shape[0] if M is None else M
    K = A.shape[1] if K is None else K
    N = B.shape[0] if N is None else N
    rc = library().fp8_gemm_blockscaled_noalloc(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(C),
                                                M, N, K, _stream(stream))
    _check(rc, "fp8_gemm_blockscaled_noalloc")
    return C


def fp8_gemm_blockscaled_residual(A, sA, B, sB, R, C, M=None, N=None, K=None, stream=None):
    """C = bf16(block-scaled GEMM + R): the residual R (bf16 [M, N], may be C
    itself) added in fp32 in the epilogue before the one bf16 rounding."""
    M = A.shape[0] if M is None else M
    K = A.shape[1] if K is None else K
    N = B.shape[0] if N is None else N
    _check(library().fp8_gemm_blockscaled_residual(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(R), _ptr(C),
                                                   M, N, K, _stream(stream)), "fp8_gemm_blockscaled_residual")
    return C


def fp8_gemm_blockscaled_quant(A, sA, B, sB, Cq, sC, M=None, N=None, K=None, stream=None):
    """(Cq, sC) = block quantization of the block-scaled GEMM's bf16 output, done
    in its epilogue: Cq E4M3 codes [M, N] (uint8 or float8 storage), sC fp32
    [ceil(M/32), N/32] scales; equal bit for bit to fp8_gemm_blockscaled
    followed by fp8_quantize_blocks."""
    M = A.shape[0] if M is None else M
    K = A.shape[1] if K is None else K
    N = B.shape[0] if N is None else N
    _check(library().fp8_gemm_blockscaled_quant(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(Cq), _ptr(sC),
                                                M, N, K, _stream(stream)), "fp8_gemm_blockscaled_quant")
    return Cq, sC


def fp8_gemm_pertoken_e8m0(A, sA, B, sB, C, M=None, N=None, K=None, stream=None):
    """C = bf16(sum_kb 2^(sA[m][kb]-127) * sB * sum_k A*B): per-token A scales as
    UE8M0 bytes (uint8 [M, K/32]), B block scales fp32 powers of two; the
    native path."""
    M = A.shape[0] if M is None else M
    K = A.shape[1] if K is None else K
    N = B.shape[0] if N is None else N
    _check(library().fp8_gemm_pertoken_e8m0(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(C), M, N, K,
                                            _stream(stream)), "fp8_gemm_pertoken_e8m0")
    return C


def fp8_gemm_rowcol(A, sA, B, sB, C, M=None, N=None, K=None, stream=None):
    """C[M,N] (bf16) = sA[m] * sB[n] * sum_k A[m,k] B[n,k]: per-token (sA, fp32
    [M]) x per-channel (sB, fp32 [N]) scales; per-tensor = constant vectors."""
    M = A.shape[0] if M is None else M
    K = A.shape[1] if K is None else K
    N = B.shape[0] if N is None else N
    _check(library().fp8_gemm_rowcol(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(C), M, N, K,
                                     _stream(stream)), "fp8_gemm_rowcol")
    return C


def fp8_gemm_pertoken(A, sA, B, sB, C, M=None, N=None, K=None, stream=None, mode=None):
    """C[M,N] (bf16) with per-token A scales: sA fp32 [M, K/32] (one per row
    of A per 32-K block), sB fp32 [N/32, K/32] blocks.  mode: None (AUTO) or
    FP8_PATH_* (NATIVE: power-of-two scales on the block-scaled MMA)."""
    M = A.shape[0] if M is None else M
    K = A.shape[1] if K is None else K
    N = B.shape[0] if N is None else N
    if mode is None:
        _check(library().fp8_gemm_pertoken(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(C), M, N, K,
                                           _stream(stream)), "fp8_gemm_pertoken")
    else:
        _check(library().fp8_gemm_pertoken_ex(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(C), M, N, K,
                                              mode, _stream(stream)), "fp8_gemm_pertoken_ex")
    return C


def fp8_quantize_blocks(x, q=None, s=None, stream=None):
    """Block quantization of bf16 activations x [M, K] (CUDA tensor) into E4M3
    codes q [M, K] (uint8) and fp32 scales s [ceil(M/32), K/32]: the A and sA
    operands of fp8_gemm_blockscaled.  Returns (q, s); allocates them when not
    given."""
    import torch
    M, K = x.shape
    if q is None:
        q = torch.empty(M, K, dtype=torch.uint8, device=x.device)
    if s is None:
        s = torch.empty((M + 31) // 32, K // 32, dtype=torch.float32, device=x.device)
    _check(library().fp8_quantize_blocks(_ptr(x), _ptr(q), _ptr(s), M, K, _stream(stream)),
           "fp8_quantize_blocks")
    return q, s


class GroupDescs:
    """The host array of per-group pointer records that fp8_gemm_grouped
    takes, built once (the tensors stay referenced) so that repeated calls on
    the same buffers skip the per-call pointer marshalling."""

    def __init__(self, groups):
        self.groups = list(groups)
        self.G = len(self.groups)
        self.arr = (fp8_group_desc * max(self.G, 1))()
        for g, (a, sa, b, sb, c) in enumerate(self.groups):
            self.arr[g] = fp8_group_desc(*[x if isinstance(x, int) else _ptr(x) for x in (a, sa, b, sb, c)])


def group_descs(groups) -> GroupDescs:
    return GroupDescs(groups)


def fp8_gemm_grouped(groups, Ms, N, K, G=None, stream=None, mode=None):
    """groups: sequence of (A_g, sA_g, B_g, sB_g, C_g) CUDA tensors (or raw
    device pointers), or a GroupDescs built from one; Ms: int32 CUDA tensor of
    G row counts (read on device)."""
    if isinstance(groups, GroupDescs):
        G = groups.G if G is None else G
        arr = groups.arr
    else:
        G = len(groups) if G is None else G
        arr = (fp8_group_desc * max(G, 1))()
        for g, (a, sa, b, sb, c) in enumerate(groups[:G]):
            arr[g] = fp8_group_desc(*[x if isinstance(x, int) else _ptr(x) for x in (a, sa, b, sb, c)])
    lib = library()
    s = _stream(stream)
    ms = Ms if isinstance(Ms, int) else _ptr(Ms)
    if mode is None:
        rc = lib.fp8_gemm_grouped(arr, ms, N, K, G, s)
    else:
        rc = lib.fp8_gemm_grouped_ex(arr, ms, N, K, G, int(mode), s)
    _check(rc, "fp8_gemm_grouped")


def group_table(groups, device):
    """The records of fp8_gemm_grouped_device: an int64 CUDA tensor [G, 5]
    holding each group's (A, sA, B, sB, C) device pointers, in the layout of
    fp8_group_desc.  The tensors must stay alive while launches use it."""
    import torch
    rows = [[x if isinstance(x, int) else _ptr(x) for x in g] for g in groups]
    return torch.tensor(rows, dtype=torch.int64).reshape(len(rows), 5).to(device)


def fp8_grouped_workspace_bytes(G: int) -> int:
    return library().fp8_grouped_workspace_bytes(int(G))


def fp8_gemm_grouped_device(table, Ms, N, K, workspace, G=None, stream=None):
    """Grouped GEMM whose records live in device memory: ``table`` is an
    int64 CUDA tensor [G, 5] of device pointers (see group_table), ``Ms`` an
    int32 CUDA tensor of row counts, ``workspace`` a CUDA tensor of at least
    fp8_grouped_workspace_bytes(G) bytes (128-byte aligned).  Every argument
    stays on the device, so a CUDA graph captured once follows later changes
    of the table and the row counts."""
    G = table.shape[0] if G is None else G
    rc = library().fp8_gemm_grouped_device(_ptr(table), _ptr(Ms), N, K, G, _ptr(workspace),
                                           workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "fp8_gemm_grouped_device")


def fp8_status_query(stream=None) -> int:
    out = ctypes.c_int(0)
    _check(library().fp8_status_query(_stream(stream), ctypes.byref(out)), "fp8_status_query")
    return out.value


def fp8_strerror(code: int) -> str:
    return library().fp8_strerror(int(code)).decode()


def fp8_version() -> int:
    return library().fp8_version()


def fp8_debug_set(key: int, value: int):
    _check(library().fp8_debug_set(int(key), int(value)), "fp8_debug_set")


def fp8_lib_shutdown():
    library().fp8_lib_shutdown()
