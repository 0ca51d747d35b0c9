"""CPU oracle for the block-scaled E4M3 GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library under
``block_scaled_fp8_sm_gb300/`` never does, and the two share no code: the
arithmetic lives in ``bsfp8_oracle.c`` (plain C, fp64), this module only builds
it with gcc and marshals numpy arrays through ctypes.

Definition followed (FP8 GEMM library article, hncyxsy.com/news/241433,
sections 2.2-2.3 and the usage example in section 6):
``C[m,n] = sum_kb sA[m//32,kb] * sB[n//32,kb] * sum_{k in kb} A[m,k]*B[n,k]``
with A [M,K] and B [N,K] E4M3 codes, sA [ceil(M/32),K/32] and sB
[ceil(N/32),K/32] fp32.  Grouped problems (same article, section 4.2: each
request of a grouped launch is its own GEMM with its own scales) are the same
routine applied per group.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsfp8_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libbsfp8_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared",
           "-ffp-contract=off", "-fno-fast-math", "-pthread",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, dp, fp, u8p = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
        lib.oracle_e4m3_table.argtypes = [dp]
        lib.oracle_e4m3_table.restype = None
        lib.oracle_e4m3_quantize.argtypes = [dp, i64, u8p]
        lib.oracle_e4m3_quantize.restype = None
        lib.oracle_bf16_rne.argtypes = [dp, i64, dp]
        lib.oracle_bf16_rne.restype = None
        lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_value.restype = ctypes.c_double
        lib.oracle_gemm.argtypes = [u8p, fp, u8p, fp, i64, i64, i64, dp, dp,
                                    ctypes.c_int, ctypes.c_int]
        lib.oracle_gemm.restype = ctypes.c_int
        lib.oracle_gemm_sampled.argtypes = [u8p, fp, u8p, fp, i64, i64, i64,
                                            dp, dp, i64, dp, dp, ctypes.c_int]
        lib.oracle_gemm_sampled.restype = ctypes.c_int
        lib.oracle_gemm_rowcol.argtypes = [u8p, fp, u8p, fp, i64, i64, i64, dp, dp]
        lib.oracle_gemm_rowcol.restype = ctypes.c_int
        lib.oracle_quantize_blocks.argtypes = [dp, i64, i64, u8p, fp]
        lib.oracle_quantize_blocks.restype = ctypes.c_int
        lib.oracle_gemm_pertoken.argtypes = [u8p, fp, u8p, fp, i64, i64, i64, dp, dp, ctypes.c_int]
        lib.oracle_gemm_pertoken.restype = ctypes.c_int
        lib.oracle_gemm_residual.argtypes = [u8p, fp, u8p, fp, dp, i64, i64, i64, dp, dp,
                                             ctypes.c_int, ctypes.c_int]
        lib.oracle_gemm_residual.restype = ctypes.c_int
        lib.oracle_gemm_residual_sampled.argtypes = [u8p, fp, u8p, fp, dp, i64, i64, i64,
                                                     dp, dp, i64, dp, dp, ctypes.c_int]
        lib.oracle_gemm_residual_sampled.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _codes(x, rows: int, K: int) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x), dtype=np.uint8)
    if a.size != rows * K:
        raise ValueError(f"expected {rows}x{K} E4M3 codes, got {a.shape}")
    return a.reshape(rows, K)


def _scales(s, rows: int, KB: int) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(s), dtype=np.float32)
    if a.size != ((rows + 31) // 32) * KB:
        raise ValueError(f"expected [{(rows + 31) // 32},{KB}] scales, got {a.shape}")
    return a.reshape((rows + 31) // 32, KB)


def e4m3_table() -> np.ndarray:
    """The 256 E4M3 code values as fp64 (NaN at 0x7F and 0xFF)."""
    out = np.empty(256, dtype=np.float64)
    _load().oracle_e4m3_table(_ptr(out))
    return out


def e4m3_quantize(x) -> np.ndarray:
    """Nearest E4M3 code, ties to even, saturating at +-448 (slow: a search)."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(a.shape, dtype=np.uint8)
    _load().oracle_e4m3_quantize(_ptr(a), a.size, _ptr(out))
    return out


def bf16_rne(x) -> np.ndarray:
    """bf16 bit patterns (uint16) of x rounded to nearest, ties to even."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(a.shape, dtype=np.uint16)
    _load().oracle_bf16_rne(_ptr(a), a.size, _ptr(out))
    return out


def bf16_value(bits) -> np.ndarray:
    """fp64 value of bf16 bit patterns."""
    b = np.asarray(bits, dtype=np.uint16)
    f = np.vectorize(lambda v: _load().oracle_bf16_value(int(v)), otypes=[np.float64])
    return f(b) if b.size else b.astype(np.float64)


def gemm(A, sA, B, sB, M: int, N: int, K: int, nthreads: int = 0,
         mutation: int = 0):
    """Reference C [M,N] and magnitude sum T [M,N], both fp64.

    ``mutation`` != 0 plants a known mistake (tests of the pins only)."""
    KB = K // 32
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    A = _codes(A, M, K)
    B = _codes(B, N, K)
    sA = _scales(sA, M, KB)
    sB = _scales(sB, N, KB)
    C = np.zeros((M, N), dtype=np.float64)
    T = np.zeros((M, N), dtype=np.float64)
    rc = _load().oracle_gemm(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), M, N, K,
                             _ptr(C), _ptr(T), int(nthreads), int(mutation))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm failed ({rc})")
    return C, T


def gemm_sampled(A, sA, B, sB, M: int, N: int, K: int, ms, ns, nthreads: int = 0):
    """Reference C and T at the sampled coordinates (ms[i], ns[i])."""
    KB = K // 32
    A = _codes(A, M, K)
    B = _codes(B, N, K)
    sA = _scales(sA, M, KB)
    sB = _scales(sB, N, KB)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    if ms.shape != ns.shape:
        raise ValueError("ms and ns differ in shape")
    C = np.zeros(ms.shape, dtype=np.float64)
    T = np.zeros(ms.shape, dtype=np.float64)
    rc = _load().oracle_gemm_sampled(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), M, N, K,
                                     _ptr(ms), _ptr(ns), ms.size,
                                     _ptr(C), _ptr(T), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_sampled failed ({rc})")
    return C, T


def grouped(A_list, sA_list, B_list, sB_list, Ms, N: int, K: int, nthreads: int = 0):
    """Per-group reference: a list of (C_g, T_g), one GEMM per group."""
    out = []
    for A, sA, B, sB, M in zip(A_list, sA_list, B_list, sB_list, Ms):
        out.append(gemm(A, sA, B, sB, int(M), N, K, nthreads))
    return out


def quantize_blocks(x_bf16_bits, M: int, K: int):
    """Block quantization of bf16 activations (x given as its uint16 bit
    patterns, [M, K]): returns (codes uint8 [M, K], scales float32
    [ceil(M/32), K/32]) with s = amax/448 per 32x32 block (1 for an all-zero
    block) and q = E4M3(x/s), fp32 division, nearest-even, saturating."""
    x = np.ascontiguousarray(np.asarray(x_bf16_bits, dtype=np.uint16).reshape(M, K))
    q = np.empty((M, K), dtype=np.uint8)
    s = np.empty(((M + 31) // 32, K // 32), dtype=np.float32)
    rc = _load().oracle_quantize_blocks(_ptr(x), M, K, _ptr(q), _ptr(s))
    if rc != 0:
        raise ValueError("oracle_quantize_blocks: bad arguments")
    return q, s


def gemm_rowcol(A, sA, B, sB, M: int, N: int, K: int):
    """Per-token x per-channel scaled GEMM: C[m,n] = sA[m]*sB[n]*sum_k A*B with
    sA [M] and sB [N] fp32 (per-tensor: constant vectors).  Returns (C, T) in
    fp64, like gemm()."""
    A = _codes(A, M, K)
    B = _codes(B, N, K)
    sA = np.ascontiguousarray(np.asarray(sA, dtype=np.float32).reshape(M))
    sB = np.ascontiguousarray(np.asarray(sB, dtype=np.float32).reshape(N))
    C = np.empty((M, N), dtype=np.float64)
    T = np.empty((M, N), dtype=np.float64)
    if _load().oracle_gemm_rowcol(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), M, N, K, _ptr(C), _ptr(T)) != 0:
        raise ValueError("oracle_gemm_rowcol: bad arguments")
    return C, T


def _bf16_bits(R, M: int, N: int) -> np.ndarray:
    a = np.asarray(R)
    if a.dtype not in (np.uint16, np.int16):
        raise ValueError(f"bf16 bit patterns must be uint16 or int16, got {a.dtype}")
    a = np.ascontiguousarray(a.view(np.uint16))
    if a.size != M * N:
        raise ValueError(f"expected {M}x{N} bf16 bit patterns, got {a.shape}")
    return a.reshape(M, N)


def gemm_residual(A, sA, B, sB, R_bits, M: int, N: int, K: int, nthreads: int = 0,
                  mutation: int = 0):
    """C = block-scaled GEMM + R with R given as bf16 bit patterns (uint16 or
    int16 [M, N]); returns (C, T) in fp64, T the GEMM's magnitude sum.
    ``mutation`` != 0 plants a known mistake (tests of the pins only)."""
    KB = K // 32
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    A = _codes(A, M, K)
    B = _codes(B, N, K)
    sA = _scales(sA, M, KB)
    sB = _scales(sB, N, KB)
    R = _bf16_bits(R_bits, M, N)
    C = np.zeros((M, N), dtype=np.float64)
    T = np.zeros((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_residual(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(R), M, N, K,
                                      _ptr(C), _ptr(T), int(nthreads), int(mutation))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_residual failed ({rc})")
    return C, T


def gemm_residual_sampled(A, sA, B, sB, R_bits, M: int, N: int, K: int, ms, ns, nthreads: int = 0):
    """gemm_residual at the sampled coordinates (ms[i], ns[i])."""
    KB = K // 32
    A = _codes(A, M, K)
    B = _codes(B, N, K)
    sA = _scales(sA, M, KB)
    sB = _scales(sB, N, KB)
    R = _bf16_bits(R_bits, M, N)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    if ms.shape != ns.shape:
        raise ValueError("ms and ns differ in shape")
    C = np.zeros(ms.shape, dtype=np.float64)
    T = np.zeros(ms.shape, dtype=np.float64)
    rc = _load().oracle_gemm_residual_sampled(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(R), M, N, K,
                                              _ptr(ms), _ptr(ns), ms.size, _ptr(C), _ptr(T), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_residual_sampled failed ({rc})")
    return C, T


def gemm_pertoken(A, sA, B, sB, M: int, N: int, K: int, mutation: int = 0):
    """Per-token A scales: C[m,n] = sum_kb sA[m,kb]*sB[n//32,kb]*sum_{k in kb}
    A[m,k]*B[n,k] with sA [M, K/32] and sB [ceil(N/32), K/32] fp32.  Returns
    (C, T) in fp64 like gemm().  ``mutation`` != 0: pin tests only."""
    KB = K // 32
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    A = _codes(A, M, K)
    B = _codes(B, N, K)
    sA = np.ascontiguousarray(np.asarray(sA, dtype=np.float32).reshape(M, KB))
    sB = _scales(sB, N, KB)
    C = np.zeros((M, N), dtype=np.float64)
    T = np.zeros((M, N), dtype=np.float64)
    if _load().oracle_gemm_pertoken(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), M, N, K,
                                    _ptr(C), _ptr(T), int(mutation)) != 0:
        raise ValueError("oracle_gemm_pertoken: bad arguments")
    return C, T
