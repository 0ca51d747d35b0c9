"""GPU parity of the per-token x per-channel scaled GEMM (fp8_gemm_rowcol,
called through the C ABI) against the CPU oracle: C[m,n] = sA[m] * sB[n] *
sum_k A[m,k] B[n,k] (FP8 GEMM library article, hncyxsy.com/news/241433,
sections 2.2-2.3).  Tolerance: tests/_accept.py."""
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


def _problem(M, N, K, seed, const=False):
    g = torch.Generator().manual_seed(seed)
    A = workloads.normal_codes(M, K, g, "cpu")
    B = workloads.normal_codes(N, K, g, "cpu")
    if const:
        sA = torch.full((M,), 0.37)
        sB = torch.full((N,), 2.5)
    else:
        sA = torch.rand(M, generator=g) * 4 - 2           # negative and positive
        sB = torch.rand(N, generator=g) * 3
        sA[0] = 0.0                                        # a zero row scale
    return A, sA.float(), B, sB.float()


def _run(bs, A, sA, B, sB, M, N, K):
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    bs.fp8_gemm_rowcol(A.to(DEV), sA.to(DEV), B.to(DEV), sB.to(DEV), C, M, N, K)
    torch.cuda.synchronize()
    return C


@pytest.mark.parametrize("M,N,K", [(1, 32, 32), (45, 96, 160), (300, 288, 1056), (256, 512, 4096)])
def test_rowcol_parity(bs, M, N, K):
    A, sA, B, sB = _problem(M, N, K, seed=M + N + K)
    C = _run(bs, A, sA, B, sB, M, N, K)
    Cr, T = oracle.gemm_rowcol(A.numpy(), sA.numpy(), B.numpy(), sB.numpy(), M, N, K)
    check(bf16_to_f64(C), Cr, T, f"rowcol {M}x{N}x{K}")
    assert torch.all(C[0] == 0)
    assert bs.fp8_status_query() == 0


def test_rowcol_per_tensor(bs):
    M, N, K = 130, 256, 512
    A, sA, B, sB = _problem(M, N, K, seed=3, const=True)
    C = _run(bs, A, sA, B, sB, M, N, K)
    Cr, T = oracle.gemm_rowcol(A.numpy(), sA.numpy(), B.numpy(), sB.numpy(), M, N, K)
    check(bf16_to_f64(C), Cr, T, "rowcol per-tensor")


def test_rowcol_full_size_rows_and_batch_invariance(bs):
    """4096^3 in the launch configuration of the square workload; whole rows
    compared with the oracle on the same rows, and the first rows bit-equal
    to an M=1 and an M=7 launch."""
    M = N = K = 4096
    A, sA, B, sB = _problem(M, N, K, seed=4)
    C = _run(bs, A, sA, B, sB, M, N, K)
    for rows in ([1, 2], [2047, 4095]):
        r = torch.tensor(rows)
        Cr, T = oracle.gemm_rowcol(A[r].numpy(), sA[r].numpy(), B.numpy(), sB.numpy(), len(rows), N, K)
        check(bf16_to_f64(C[r.to(DEV)]), Cr, T, f"rowcol 4096^3 rows {rows}")
    for m in (1, 7):
        Cm = _run(bs, A[:m].contiguous(), sA[:m].contiguous(), B, sB, m, N, K)
        assert torch.equal(Cm.view(torch.int16), C[:m].view(torch.int16)), f"M={m}"
