"""GPU parity of the block-scaled GEMM with a fused residual add
(fp8_gemm_blockscaled_residual, through the C ABI): C = bf16(GEMM + R)
against the oracle's GEMM + residual (oracle_gemm_residual), element by
element.  Tolerance: tests/_accept.py with the GEMM's magnitude sum T (R is
exact in fp32 and adds one rounding).  Besides small and ragged shapes, the
4096^3 problem the benchmark times (256 tiles on 76 CTA pairs, so every CTA
runs several tiles and reuses its residual staging buffer) is compared on
sampled elements and whole rows, out of place and in place, on both paths."""
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
    return oracle.gemm_residual(A.numpy(), sA.numpy(), B.numpy(), sB.numpy(),
                                R.view(torch.int16).numpy(), M, N, K)


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


# ------------------------------------------------- multi-tile (bench size)

def _bench_size_problem(arbitrary):
    """The 4096^3 square workload (power-of-two scales), or the same codes
    with arbitrary fp32 scales (every tile promotes), plus a seeded bf16
    residual; generated on the device like the benchmark's inputs."""
    p = workloads.make("c1", seed=0, device=DEV)
    if arbitrary:
        g = torch.Generator(device=DEV).manual_seed(7)
        p.sA = torch.rand(p.sA.shape, generator=g, device=DEV) * 2 + 0.05
        p.sB = torch.rand(p.sB.shape, generator=g, device=DEV) * 2 + 0.05
    g = torch.Generator(device=DEV).manual_seed(1)
    R = torch.randn(p.M, p.N, generator=g, device=DEV).to(torch.bfloat16)
    return p, R


def _sampled_residual_check(p, R, C, what, n_samples=6000):
    rng = np.random.default_rng(3)
    rows = (0, 255, 256, p.M - 1)
    ms = np.concatenate([rng.integers(0, p.M, n_samples)] + [np.full(p.N, r) for r in rows])
    ns = np.concatenate([rng.integers(0, p.N, n_samples)] + [np.arange(p.N) for _ in rows])
    A, sA, B, sB = (t.cpu().numpy() for t in (p.A, p.sA, p.B, p.sB))
    Cr, T = oracle.gemm_residual_sampled(A, sA, B, sB, R.cpu().view(torch.int16).numpy(),
                                         p.M, p.N, p.K, ms, ns)
    Cg = C[torch.from_numpy(ms).to(DEV), torch.from_numpy(ns).to(DEV)]
    check(bf16_to_f64(Cg), Cr, T, what)


@pytest.mark.parametrize("arbitrary", [False, True])
def test_residual_bench_size_multi_tile(bs, arbitrary):
    p, R = _bench_size_problem(arbitrary)
    buf = torch.full((p.M + 2, p.N), -7.0, dtype=torch.bfloat16, device=DEV)
    C = buf[1:p.M + 1]
    bs.fp8_gemm_blockscaled_residual(p.A, p.sA, p.B, p.sB, R, C, p.M, p.N, p.K)
    torch.cuda.synchronize()
    assert torch.all(buf[0] == -7.0) and torch.all(buf[-1] == -7.0), "store outside C"
    assert bs.fp8_status_query() == 0
    _sampled_residual_check(p, R, C, f"residual 4096^3{' arb' if arbitrary else ''}")


@pytest.mark.parametrize("arbitrary", [False, True])
def test_residual_bench_size_in_place(bs, arbitrary):
    p, R = _bench_size_problem(arbitrary)
    C = R.clone()
    bs.fp8_gemm_blockscaled_residual(p.A, p.sA, p.B, p.sB, C, C, p.M, p.N, p.K)
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == 0
    _sampled_residual_check(p, R, C, f"residual 4096^3 in place{' arb' if arbitrary else ''}")
    # in place and out of place give the same bits
    C2 = torch.empty_like(C)
    bs.fp8_gemm_blockscaled_residual(p.A, p.sA, p.B, p.sB, R, C2, p.M, p.N, p.K)
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16), C2.view(torch.int16))
