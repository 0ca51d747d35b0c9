"""The allocation-free entry point against the regular one.

fp8_gemm_blockscaled_noalloc serves callers that cannot allocate device
memory (for example a server whose caching allocator owns the whole GPU, or a
deployment whose memory budget is fixed at start-up): its only scratch, the
kernel's status word, is a static array inside the library, and
fp8_status_query reads that word back without allocating either.  The two
entry points run different tile heights (128-row single-CTA tiles against
256-row CTA pairs) with the same per-element arithmetic, so with scales whose
row blocks are all of one kind their outputs agree bit for bit.

This file is collected last so that a run stopping at the first failure has
already run every other test; it passes on its own in a fresh process too.
"""
import pytest
import torch

import oracle
from tests._accept import bf16_to_f64, check

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def bs():
    import block_scaled_fp8_sm_gb300 as mod
    from block_scaled_fp8_sm_gb300 import build
    build.build()
    mod.library()
    return mod


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
def test_noalloc_matches_regular_entry_point_twice(bs, pow2):
    lib = bs.library()
    for call, (M, N, K) in enumerate([(200, 512, 416), (129, 256, 1024)]):
        A, sA, B, sB = _problem(M, N, K, seed=31 + call + (0 if pow2 else 100), pow2=pow2)
        c_new = _call(lib.fp8_gemm_blockscaled_noalloc, A, sA, B, sB, M, N, K)
        c_old = _call(lib.fp8_gemm_blockscaled, A, sA, B, sB, M, N, K)
        # every row block of sA is of one kind here, so both entry points take
        # the same path for every element: the same bits
        assert torch.equal(c_new.view(torch.int16), c_old.view(torch.int16)), f"call {call}"
        Cr, T = oracle.gemm(A.numpy(), sA.numpy(), B.numpy(), sB.numpy(), M, N, K)
        check(bf16_to_f64(c_new), Cr, T, f"noalloc call {call}{'' if pow2 else ' arb'}")
    assert bs.fp8_status_query() == 0


def test_noalloc_wait_timeout_is_reported(bs):
    """A withheld pipeline stage makes the allocation-free call's waits run
    out; the condition lands in the static status word and fp8_status_query
    reports it (and clears it), and the next call is correct."""
    lib = bs.library()
    M, N, K = 512, 512, 512
    A, sA, B, sB = _problem(M, N, K, seed=7, pow2=True)
    assert bs.fp8_status_query() == 0
    bs.fp8_debug_set(bs.FP8_DEBUG_WAIT_LIMIT_CYCLES, 20_000_000)   # ~10 ms
    bs.fp8_debug_set(bs.FP8_DEBUG_WITHHOLD_STAGE, 1)
    try:
        _call(lib.fp8_gemm_blockscaled_noalloc, A, sA, B, sB, M, N, K)
        assert bs.fp8_status_query() == bs._abi.FP8_ERR_TIMEOUT
    finally:
        bs.fp8_debug_set(bs.FP8_DEBUG_WITHHOLD_STAGE, -1)
        bs.fp8_debug_set(bs.FP8_DEBUG_WAIT_LIMIT_CYCLES, 0)
    assert bs.fp8_status_query() == 0   # read and cleared
    C = _call(lib.fp8_gemm_blockscaled_noalloc, A, sA, B, sB, M, N, K)
    assert bs.fp8_status_query() == 0
    Cr, T = oracle.gemm(A.numpy(), sA.numpy(), B.numpy(), sB.numpy(), M, N, K)
    check(bf16_to_f64(C), Cr, T, "noalloc after timeout")


def test_noalloc_argument_errors(bs):
    lib = bs.library()
    assert lib.fp8_gemm_blockscaled_noalloc(16, 16, 16, 16, 16, 64, 33, 64, None) == -2
    assert lib.fp8_gemm_blockscaled_noalloc(16, 16, 16, 16, 0, 64, 64, 64, None) == -1
    assert lib.fp8_gemm_blockscaled_noalloc(0, 0, 0, 0, 0, 0, 64, 64, None) == 0
