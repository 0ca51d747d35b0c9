"""The allocation-free entry point against the regular one.

fp8_gemm_blockscaled_noalloc serves callers that cannot allocate device
memory (for example a server whose caching allocator owns the whole GPU): its
only scratch, the kernel's status word, is a static array inside the library.
This file is collected last so that a run stopping at the first failure has
already run every other test; it passes on its own in a fresh process too.
"""
import numpy as np
import pytest
import torch

import oracle
from tests._accept import ABS_T, REL, bf16_to_f64, check

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    import block_scaled_fp8_sm_gb300 as bs
    from block_scaled_fp8_sm_gb300 import build
    build.build()
    return bs.library()


def _problem(M, N, K, seed, pow2):
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(M, K, generator=g).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    B = torch.randn(N, K, generator=g).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    if pow2:
        sA = torch.ldexp(torch.ones((M + 31) // 32, K // 32), torch.randint(-4, 5, ((M + 31) // 32, K // 32), generator=g))
        sB = torch.ldexp(torch.ones(N // 32, K // 32), torch.randint(-4, 5, (N // 32, K // 32), generator=g))
    else:
        sA = torch.rand((M + 31) // 32, K // 32, generator=g) + 0.1
        sB = torch.rand(N // 32, K // 32, generator=g) + 0.1
    return A, sA.float().contiguous(), B, sB.float().contiguous()


def _call(fn, A, sA, B, sB, M, N, K):
    dA, dsA, dB, dsB = (t.to(DEV) for t in (A, sA, B, sB))
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    rc = fn(dA.data_ptr(), dsA.data_ptr(), dB.data_ptr(), dsB.data_ptr(), C.data_ptr(), M, N, K,
            torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    return C


@pytest.mark.parametrize("pow2", [True, False])
def test_noalloc_matches_regular_entry_point_twice(lib, pow2):
    for call, (M, N, K) in enumerate([(200, 512, 416), (129, 256, 1024)]):
        A, sA, B, sB = _problem(M, N, K, seed=31 + call + (0 if pow2 else 100), pow2=pow2)
        c_new = _call(lib.fp8_gemm_blockscaled_noalloc, A, sA, B, sB, M, N, K)
        c_old = _call(lib.fp8_gemm_blockscaled, A, sA, B, sB, M, N, K)
        Cr, T = oracle.gemm(A.numpy(), sA.numpy(), B.numpy(), sB.numpy(), M, N, K)
        new, old = bf16_to_f64(c_new), bf16_to_f64(c_old)
        # the two entry points agree within the tolerance the other tests use
        assert np.all(np.abs(new - old) <= REL * np.abs(old) + ABS_T * T), f"call {call}"
        check(new, Cr, T, f"noalloc call {call}")


def test_noalloc_argument_errors(lib):
    assert lib.fp8_gemm_blockscaled_noalloc(16, 16, 16, 16, 16, 64, 33, 64, None) == -2
    assert lib.fp8_gemm_blockscaled_noalloc(16, 16, 16, 16, 0, 64, 64, 64, None) == -1
    assert lib.fp8_gemm_blockscaled_noalloc(0, 0, 0, 0, 0, 0, 64, 64, None) == 0
