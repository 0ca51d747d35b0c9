"""GPU parity of the block-scaled GEMM with a fused residual add
(fp8_gemm_blockscaled_residual, through the C ABI): C = bf16(GEMM + R), the
GEMM from the CPU oracle and R added in fp64.  Tolerance: tests/_accept.py
with the GEMM's magnitude sum T (R is exact in fp32 and adds one rounding)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
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


def _problem(M, N, K, seed, arbitrary=False):
    g = torch.Generator().manual_seed(seed)
    A = workloads.normal_codes(M, K, g, "cpu")
    B = workloads.normal_codes(N, K, g, "cpu")
    if arbitrary:
        sA = torch.rand((M + 31) // 32, K // 32, generator=g) * 2 + 0.05
        sB = torch.rand(N // 32, K // 32, generator=g) * 2 + 0.05
    else:
        sA = workloads.pow2_scales(M, K // 32, -4, 4, g, "cpu")
        sB = workloads.pow2_scales(N, K // 32, -4, 4, g, "cpu")
    R = (torch.randn(M, N, generator=g) * 20).to(torch.bfloat16)
    return A, sA, B, sB, R


def _expected(A, sA, B, sB, R, M, N, K):
    Cr, T = oracle.gemm(A.numpy(), sA.numpy(), B.numpy(), sB.numpy(), M, N, K)
    return Cr + R.float().numpy().astype(np.float64), T


@pytest.mark.parametrize("M,N,K,arbitrary", [(1, 32, 64, False), (77, 288, 544, False), (300, 512, 1024, False),
                                             (129, 256, 256, True)])
def test_residual_parity(bs, M, N, K, arbitrary):
    A, sA, B, sB, R = _problem(M, N, K, seed=M + K, arbitrary=arbitrary)
    buf = torch.full((M + 2, N), -7.0, dtype=torch.bfloat16, device=DEV)   # guard rows around C
    C = buf[1:M + 1]
    bs.fp8_gemm_blockscaled_residual(A.to(DEV), sA.to(DEV), B.to(DEV), sB.to(DEV), R.to(DEV), C, M, N, K)
    torch.cuda.synchronize()
    assert torch.all(buf[0] == -7.0) and torch.all(buf[-1] == -7.0), "store outside C"
    exp, T = _expected(A, sA, B, sB, R, M, N, K)
    check(bf16_to_f64(C), exp, T, f"residual {M}x{N}x{K}{' arb' if arbitrary else ''}")
    assert bs.fp8_status_query() == 0


def test_residual_in_place_and_k_zero(bs):
    M, N, K = 200, 256, 768
    A, sA, B, sB, R = _problem(M, N, K, seed=5)
    C = R.to(DEV).clone()
    bs.fp8_gemm_blockscaled_residual(A.to(DEV), sA.to(DEV), B.to(DEV), sB.to(DEV), C, C, M, N, K)
    torch.cuda.synchronize()
    exp, T = _expected(A, sA, B, sB, R, M, N, K)
    check(bf16_to_f64(C), exp, T, "residual in place")
    C0 = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    e = torch.empty(0, dtype=torch.uint8, device=DEV)
    f = torch.empty(0, dtype=torch.float32, device=DEV)
    bs.fp8_gemm_blockscaled_residual(e, f, e, f, R.to(DEV), C0, M, N, 0)
    torch.cuda.synchronize()
    assert torch.equal(C0.cpu().view(torch.int16), R.view(torch.int16))


def test_residual_zero_equals_plain_bits(bs):
    """With R = 0 the fused call gives exactly the plain call's bits."""
    M, N, K = 256, 512, 2048
    A, sA, B, sB, _ = _problem(M, N, K, seed=6)
    d = [t.to(DEV) for t in (A, sA, B, sB)]
    C1 = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    C2 = torch.empty_like(C1)
    bs.fp8_gemm_blockscaled(*d, C1, M, N, K)
    bs.fp8_gemm_blockscaled_residual(*d, torch.zeros(M, N, dtype=torch.bfloat16, device=DEV), C2, M, N, K)
    torch.cuda.synchronize()
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))
