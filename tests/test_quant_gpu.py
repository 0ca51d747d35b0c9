"""GPU parity of the block quantizer (fp8_quantize_blocks, called through the
C ABI) against the CPU oracle: codes and scales bit-exact (the code is an
integer decided by fp32 arithmetic on both sides)."""
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


def _activations(M, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, K, generator=g)
    x = torch.where(torch.rand(M, K, generator=g) < 0.005, x * 50.0, x)   # outliers
    x[:, :32] *= 1e-4                                                    # subnormal codes
    if M > 40 and K > 64:
        x[32:64, 32:64] = 0.0                                            # an all-zero block
        x[33, 40] = -0.0
    return x.to(torch.bfloat16)


def _bits(xb):
    return xb.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("M,K", [(1, 32), (31, 96), (33, 288), (77, 512), (300, 256), (64, 2080)])
def test_quantize_bit_exact(bs, M, K):
    xb = _activations(M, K, seed=M * 7 + K)
    q, s = bs.fp8_quantize_blocks(xb.to(DEV))
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_blocks(_bits(xb), M, K)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q_ref)


def test_quantize_full_size_sampled_strips(bs):
    """8192 x 8192 activations (the arbitrary-scale workload's A), with the
    launch configuration the bench times; 32-row strips compared whole."""
    M = K = 8192
    xb = _activations(M, K, seed=5)
    q, s = bs.fp8_quantize_blocks(xb.to(DEV))
    torch.cuda.synchronize()
    for mb in (0, 1, 127, 255):
        rows = slice(32 * mb, 32 * mb + 32)
        q_ref, s_ref = oracle.quantize_blocks(_bits(xb[rows].contiguous()), 32, K)
        assert np.array_equal(s[mb].cpu().numpy().view(np.uint32), s_ref[0].view(np.uint32)), f"strip {mb}"
        assert np.array_equal(q[rows].cpu().numpy(), q_ref), f"strip {mb}"


def test_quantized_operands_feed_the_gemm(bs):
    """The codes and scales are the GEMM's A and sA: quantize, multiply, and
    compare with the oracle GEMM of the oracle's own quantization."""
    M, N, K = 100, 96, 320
    xb = _activations(M, K, seed=9)
    q, s = bs.fp8_quantize_blocks(xb.to(DEV))
    g = torch.Generator().manual_seed(10)
    B = workloads.normal_codes(N, K, g, "cpu")
    sB = workloads.pow2_scales(N, K // 32, -4, 4, g, "cpu")
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    bs.fp8_gemm_blockscaled(q, s, B.to(DEV), sB.to(DEV), C, M, N, K)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_blocks(_bits(xb), M, K)
    Cr, T = oracle.gemm(q_ref, s_ref, B.numpy(), sB.numpy(), M, N, K)
    check(bf16_to_f64(C), Cr, T, "quantize -> gemm")
