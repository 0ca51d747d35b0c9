"""GPU parity of the block-scaled GEMM with its output quantized in the
epilogue (fp8_gemm_blockscaled_quant, through the C ABI).  Its contract is
the chain of two existing calls, bit for bit: fp8_gemm_blockscaled (whose bf16
output is pinned to the oracle's GEMM elsewhere) followed by
fp8_quantize_blocks.  Each case checks the codes and scales against (1) that
chain on the GPU and (2) the oracle's block quantizer applied to the GPU GEMM's
bf16 output, so the quantization arithmetic is pinned to the oracle directly.
Shapes: single blocks, ragged M and N (the last 32-row block partial, the last
tile cut), several K stages, power-of-two scales (native tiles) and arbitrary
ones (promotion tiles), and the 4096^3 problem where every CTA pair runs
several tiles."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def bs():
    import block_scaled_fp8_sm_gb300 as mod
    from block_scaled_fp8_sm_gb300 import build
    build.build()
    mod.library()
    return mod


def _problem(M, N, K, seed, arbitrary):
    g = torch.Generator().manual_seed(seed)
    A = workloads.normal_codes(M, K, g, "cpu")
    B = workloads.normal_codes(N, K, g, "cpu")
    if arbitrary:
        sA = torch.rand((M + 31) // 32, K // 32, generator=g) * 2 + 0.05
        sB = torch.rand(N // 32, K // 32, generator=g) * 2 + 0.05
    else:
        sA = workloads.pow2_scales(M, K // 32, -4, 4, g, "cpu")
        sB = workloads.pow2_scales(N, K // 32, -4, 4, g, "cpu")
    return A.to(DEV), sA.to(DEV), B.to(DEV), sB.to(DEV)


def _fused(bs, A, sA, B, sB, M, N, K):
    # guard rows around the codes and a guard row after the scales catch stray stores
    qbuf = torch.full((M + 2, N), 0xA5, dtype=torch.uint8, device=DEV)
    sbuf = torch.full(((M + 31) // 32 + 1, N // 32), -3.0, dtype=torch.float32, device=DEV)
    Cq, sC = qbuf[1:M + 1], sbuf[:(M + 31) // 32]
    bs.fp8_gemm_blockscaled_quant(A, sA, B, sB, Cq, sC, M, N, K)
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == 0
    assert torch.all(qbuf[0] == 0xA5) and torch.all(qbuf[-1] == 0xA5), "code store outside Cq"
    assert torch.all(sbuf[-1] == -3.0), "scale store outside sC"
    return Cq, sC


def _chain(bs, A, sA, B, sB, M, N, K):
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    bs.fp8_gemm_blockscaled(A, sA, B, sB, C, M, N, K)
    q, s = bs.fp8_quantize_blocks(C)
    torch.cuda.synchronize()
    return C, q, s


def _same(a, b):
    return np.array_equal(a.cpu().numpy().view(np.uint8), b.cpu().numpy().view(np.uint8))


@pytest.mark.parametrize("M,N,K,arbitrary", [(1, 32, 32, False), (32, 32, 64, False), (45, 96, 160, False),
                                             (300, 288, 1056, False), (256, 512, 2048, False),
                                             (77, 256, 512, True), (300, 288, 1056, True)])
def test_quant_out_equals_chain_and_oracle(bs, M, N, K, arbitrary):
    A, sA, B, sB = _problem(M, N, K, seed=M * 3 + N + K, arbitrary=arbitrary)
    Cq, sC = _fused(bs, A, sA, B, sB, M, N, K)
    C, q, s = _chain(bs, A, sA, B, sB, M, N, K)
    assert _same(Cq, q), f"codes differ from the GEMM + quantizer chain ({M}x{N}x{K})"
    assert _same(sC, s), f"scales differ from the GEMM + quantizer chain ({M}x{N}x{K})"
    q_ref, s_ref = oracle.quantize_blocks(C.cpu().view(torch.int16).numpy().view(np.uint16), M, N)
    assert np.array_equal(Cq.cpu().numpy(), q_ref), "codes differ from the oracle's quantizer"
    assert np.array_equal(sC.cpu().numpy().view(np.uint32), s_ref.view(np.uint32)), "scales differ from the oracle's"


def test_quant_out_4096_multi_tile(bs):
    """4096^3: 256 tiles on 76 CTA pairs, every pair runs several tiles; whole
    output against the chain, four 32-row strips against the oracle."""
    M = N = K = 4096
    A, sA, B, sB = _problem(M, N, K, seed=11, arbitrary=False)
    Cq, sC = _fused(bs, A, sA, B, sB, M, N, K)
    C, q, s = _chain(bs, A, sA, B, sB, M, N, K)
    assert _same(Cq, q) and _same(sC, s)
    for mb in (0, 1, 64, 127):
        rows = slice(32 * mb, 32 * mb + 32)
        q_ref, s_ref = oracle.quantize_blocks(C[rows].cpu().contiguous().view(torch.int16).numpy().view(np.uint16), 32, N)
        assert np.array_equal(Cq[rows].cpu().numpy(), q_ref), f"strip {mb}"
        assert np.array_equal(sC[mb:mb + 1].cpu().numpy().view(np.uint32), s_ref.view(np.uint32)), f"strip {mb}"


def test_quant_out_block_invariance(bs):
    """A 32-row block's codes and scale do not depend on M beyond that block."""
    N, K = 512, 1024
    A, sA, B, sB = _problem(512, N, K, seed=5, arbitrary=False)
    ref_q, ref_s = _fused(bs, A, sA, B, sB, 512, N, K)
    for M in (32, 96, 288):
        Cq, sC = _fused(bs, A[:M].contiguous(), sA[:M // 32].contiguous(), B, sB, M, N, K)
        assert _same(Cq, ref_q[:M]) and _same(sC, ref_s[:M // 32]), f"M={M}"


def test_quant_out_k_zero(bs):
    """K = 0: C = 0, so every block is all zero: codes 0 and scales 1."""
    M, N = 40, 64
    qbuf = torch.full((M, N), 0x5A, dtype=torch.uint8, device=DEV)
    sbuf = torch.full(((M + 31) // 32, N // 32), -3.0, dtype=torch.float32, device=DEV)
    A = torch.empty(M, 0, dtype=torch.uint8, device=DEV)
    B = torch.empty(N, 0, dtype=torch.uint8, device=DEV)
    bs.fp8_gemm_blockscaled_quant(A, sbuf, B, sbuf, qbuf, sbuf, M, N, 0)
    torch.cuda.synchronize()
    assert torch.all(qbuf == 0) and torch.all(sbuf == 1.0)
