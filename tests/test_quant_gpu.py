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


def test_quantize_rounding_midpoints(bs):
    """Quotients x / s that are E4M3 rounding midpoints (exact ties, which
    round to the even code) or lie just above one, with scales whose
    reciprocal is inexact (s = 3, 5, 7, 1.5): a reciprocal product instead of
    the correctly rounded division would give 234 wrong codes on this data."""
    rng = np.random.default_rng(21)
    # E4M3 midpoints: normal (1 + (2j+1)/16) * 2^e, e in [-6, 8], and subnormal (2j+1) * 2^-10
    mids = [(1 + (2 * j + 1) / 16) * 2.0 ** e for e in range(-6, 8) for j in range(8)]
    mids += [(2 * j + 1) * 2.0 ** -10 for j in range(8)]
    mids = np.array(mids)
    blocks = []
    for k in (3.0, 5.0, 7.0, 1.5):
        blk = np.empty((32, 32))
        vals = rng.choice(mids, size=32 * 32) * k * rng.choice([-1.0, 1.0], size=32 * 32)
        blk[:] = vals.reshape(32, 32)
        blk[0, 0] = 448.0 * k                      # the block maximum: s = k exactly
        blocks.append(blk)
    x = torch.from_numpy(np.concatenate(blocks, axis=1)).to(torch.float32)   # 32 x 128
    xb = x.to(torch.bfloat16)
    # the chosen values are exact in bf16 (few significant bits), so x / s are the midpoints
    assert torch.equal(xb.to(torch.float32), x)
    # neighbours one bf16 step away: quotients just off the midpoints
    up = (xb.view(torch.int16) + 1).view(torch.bfloat16)
    both = torch.cat([xb, up], dim=0)                                       # 64 x 128
    both[32, 0] = xb[0, 0]
    both[32, 32] = xb[0, 32]
    both[32, 64] = xb[0, 64]
    both[32, 96] = xb[0, 96]
    M, K = both.shape
    q, s = bs.fp8_quantize_blocks(both.to(DEV))
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_blocks(_bits(both.contiguous()), M, K)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q_ref)


def test_quantize_wide_exponents_and_subnormal_scales(bs):
    """Every block gets its own maximum, from 2^-133 (a bf16 subnormal, whose
    scale amax/448 is an fp32 subnormal) up to 2^120, and random bf16 values
    below it, zeros and negative zeros included: the codes and scales match
    the oracle's fp32 division bit for bit on both sides of the normal-scale
    boundary."""
    rng = np.random.default_rng(33)
    MB, KB = 8, 64                                   # 512 blocks of 32 x 32
    exps = np.linspace(-133, 120, MB * KB).round().astype(int)
    rng.shuffle(exps)
    x = np.empty((MB * 32, KB * 32), dtype=np.float32)
    for b, e in enumerate(exps):
        mb, kb = divmod(b, KB)
        amax = np.float32(2.0 ** e) * np.float32(rng.uniform(1.0, 2.0))
        blk = rng.uniform(-1.0, 1.0, size=(32, 32)).astype(np.float32) * amax
        blk[0, 0] = amax
        blk[1, 1] = 0.0
        blk[2, 2] = -0.0
        x[mb * 32:(mb + 1) * 32, kb * 32:(kb + 1) * 32] = blk
    xb = torch.from_numpy(x).to(torch.bfloat16)
    M, K = xb.shape
    q, s = bs.fp8_quantize_blocks(xb.to(DEV))
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_blocks(_bits(xb.contiguous()), M, K)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert (s_ref < np.float32(1.17549435e-38)).any() and (s_ref > 1.0).any()
