"""GPU parity of the GEMM with per-token A scales (fp8_gemm_pertoken, through
the C ABI): one fp32 scale per row of A per 32-K block, B with 32x32 blocks
(FP8 GEMM library article, hncyxsy.com/news/241433, section 2.2), against
the oracle's oracle_gemm_pertoken element by element; the block-constant
case against the block-scaled call bit for bit; rows bit-identical across M."""
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


def _problem(M, N, K, seed, pow2=False):
    g = torch.Generator().manual_seed(seed)
    A = workloads.normal_codes(M, K, g, "cpu")
    B = workloads.normal_codes(N, K, g, "cpu")
    if pow2:
        sA = torch.ldexp(torch.ones(M, K // 32), torch.randint(-4, 5, (M, K // 32), generator=g)).float()
        sB = workloads.pow2_scales(N, K // 32, -4, 4, g, "cpu")
    else:
        sA = torch.rand(M, K // 32, generator=g) * 2 + 0.05
        sB = torch.rand(N // 32, K // 32, generator=g) * 2 + 0.05
    return A, sA.contiguous(), B, sB.contiguous()


def _run(bs, A, sA, B, sB, M, N, K):
    buf = torch.full((M + 2, N), -7.0, dtype=torch.bfloat16, device=DEV)
    C = buf[1:M + 1]
    bs.fp8_gemm_pertoken(A.to(DEV), sA.to(DEV), B.to(DEV), sB.to(DEV), C, M, N, K)
    torch.cuda.synchronize()
    assert torch.all(buf[0] == -7.0) and torch.all(buf[-1] == -7.0), "store outside C"
    return C


@pytest.mark.parametrize("M,N,K,pow2", [(1, 32, 32, False), (45, 96, 160, False), (130, 288, 480, True),
                                        (300, 512, 1056, False), (257, 256, 2048, True)])
def test_pertoken_parity(bs, M, N, K, pow2):
    A, sA, B, sB = _problem(M, N, K, seed=M + N + K, pow2=pow2)
    C = _run(bs, A, sA, B, sB, M, N, K)
    Cr, T = oracle.gemm_pertoken(A.numpy(), sA.numpy(), B.numpy(), sB.numpy(), M, N, K)
    check(bf16_to_f64(C), Cr, T, f"pertoken {M}x{N}x{K}{' pow2' if pow2 else ''}")
    assert bs.fp8_status_query() == 0


def test_block_constant_scales_equal_the_block_scaled_promotion(bs):
    M, N, K = 1000, 512, 1024
    A, _, B, sB = _problem(M, N, K, seed=5)
    g = torch.Generator().manual_seed(6)
    sA_blk = torch.rand((M + 31) // 32, K // 32, generator=g) + 0.1
    sA_tok = sA_blk.repeat_interleave(32, dim=0)[:M].contiguous()
    C_tok = _run(bs, A, sA_tok, B, sB, M, N, K)
    C_blk = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    bs.fp8_gemm_blockscaled(A.to(DEV), sA_blk.to(DEV), B.to(DEV), sB.to(DEV), C_blk, M, N, K, mode=bs.FP8_PATH_PROMOTE)
    torch.cuda.synchronize()
    assert torch.equal(C_tok.view(torch.int16), C_blk.view(torch.int16))


def test_pertoken_batch_invariance(bs):
    M, N, K = 4096, 512, 1024
    A, sA, B, sB = _problem(M, N, K, seed=7)
    dB, dsB = B.to(DEV), sB.to(DEV)
    rows = {}
    for m in (1, 7, 64, M):
        C = torch.empty(m, N, dtype=torch.bfloat16, device=DEV)
        bs.fp8_gemm_pertoken(A[:m].contiguous().to(DEV), sA[:m].contiguous().to(DEV), dB, dsB, C, m, N, K)
        torch.cuda.synchronize()
        rows[m] = C[:64].view(torch.int16).cpu()
    for m in (1, 7, 64):
        k = min(m, 64)
        assert torch.equal(rows[m][:k], rows[M][:k]), f"M={m}"
    Cr, T = oracle.gemm_pertoken(A[:64].numpy(), sA[:64].numpy(), B.numpy(), sB.numpy(), 64, N, K)
    check(bf16_to_f64(rows[M].view(torch.bfloat16)), Cr, T, "pertoken batch invariance rows")


def test_pertoken_square_4096_sampled(bs):
    M = N = K = 4096
    g = torch.Generator(device=DEV).manual_seed(8)
    A = workloads.normal_codes(M, K, g, DEV)
    B = workloads.normal_codes(N, K, g, DEV)
    sA = torch.rand(M, K // 32, generator=g, device=DEV) + 0.05
    sB = torch.rand(N // 32, K // 32, generator=g, device=DEV) + 0.05
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    bs.fp8_gemm_pertoken(A, sA, B, sB, C, M, N, K)
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == 0
    rng = np.random.default_rng(8)
    rows = np.unique(np.concatenate([[0, 127, 128, 2049, M - 1], rng.integers(0, M, 60)]))
    Ah, sAh, Bh, sBh = (t.cpu().numpy() for t in (A, sA, B, sB))
    Cr, T = oracle.gemm_pertoken(Ah[rows], sAh[rows], Bh, sBh, len(rows), N, K)   # whole rows
    Cg = C[torch.from_numpy(rows).to(DEV)]
    check(bf16_to_f64(Cg), Cr, T, "pertoken 4096^3 rows")


# ------------------------------------------------------------- native path
# FP8_PATH_NATIVE: power-of-two per-token scales on the block-scaled MMA, every
# row of A with its own UE8M0 scale per 32-K block.

def _run_native(bs, A, sA, B, sB, M, N, K):
    buf = torch.full((M + 2, N), -7.0, dtype=torch.bfloat16, device=DEV)
    C = buf[1:M + 1]
    bs.fp8_gemm_pertoken(A.to(DEV), sA.to(DEV), B.to(DEV), sB.to(DEV), C, M, N, K, mode=bs.FP8_PATH_NATIVE)
    torch.cuda.synchronize()
    assert torch.all(buf[0] == -7.0) and torch.all(buf[-1] == -7.0), "store outside C"
    return C


@pytest.mark.parametrize("M,N,K", [(1, 256, 256), (77, 256, 160), (256, 512, 1024), (300, 288, 2048),
                                   (1000, 768, 1056)])
def test_pertoken_native_parity(bs, M, N, K):
    """Every row has its own scales (e uniform in [-4, 4] per row and K block):
    a wrong row-to-line mapping would scale rows by other rows' factors.  K=160
    and 1056 end inside a 128-K half; N=288 ends inside a 256-column tile."""
    A, sA, B, sB = _problem(M, N, K, seed=11 * M + N + K, pow2=True)
    C = _run_native(bs, A, sA, B, sB, M, N, K)
    Cr, T = oracle.gemm_pertoken(A.numpy(), sA.numpy(), B.numpy(), sB.numpy(), M, N, K)
    check(bf16_to_f64(C), Cr, T, f"pertoken native {M}x{N}x{K}")
    assert bs.fp8_status_query() == 0


def test_pertoken_native_block_constant_equals_block_scaled_native(bs):
    """Scales equal within each 32-row block: the per-row lines hold the values
    the block-scaled call replicates, so the two launches agree bit for bit."""
    M, N, K = 1000, 512, 1024
    A, _, B, sB = _problem(M, N, K, seed=12, pow2=True)
    g = torch.Generator().manual_seed(13)
    sA_blk = workloads.pow2_scales(M, K // 32, -4, 4, g, "cpu")   # [ceil(M/32), K/32]
    assert sA_blk.shape == ((M + 31) // 32, K // 32)
    sA_tok = sA_blk.repeat_interleave(32, dim=0)[:M].contiguous()
    assert sA_tok.shape == (M, K // 32)
    C_tok = _run_native(bs, A, sA_tok, B, sB, M, N, K)
    C_blk = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    bs.fp8_gemm_blockscaled(A.to(DEV), sA_blk.to(DEV), B.to(DEV), sB.to(DEV), C_blk, M, N, K,
                            mode=bs.FP8_PATH_NATIVE)
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == 0
    assert torch.equal(C_tok.view(torch.int16), C_blk.view(torch.int16))


def test_pertoken_native_batch_invariance(bs):
    M, N, K = 4096, 512, 1024
    A, sA, B, sB = _problem(M, N, K, seed=14, pow2=True)
    dB, dsB = B.to(DEV), sB.to(DEV)
    rows = {}
    for m in (1, 7, 64, M):
        C = torch.empty(m, N, dtype=torch.bfloat16, device=DEV)
        bs.fp8_gemm_pertoken(A[:m].contiguous().to(DEV), sA[:m].contiguous().to(DEV), dB, dsB, C, m, N, K,
                             mode=bs.FP8_PATH_NATIVE)
        torch.cuda.synchronize()
        rows[m] = C[:min(m, 64)].cpu()
    for m in (7, 64, M):
        n = min(m, 64)
        assert torch.equal(rows[m][:n].view(torch.int16), rows[M][:n].view(torch.int16)), m
    assert torch.equal(rows[1].view(torch.int16), rows[M][:1].view(torch.int16))
    assert bs.fp8_status_query() == 0


@pytest.mark.parametrize("which", ["sA", "sB"])
def test_pertoken_native_reports_a_scale_that_is_not_a_power_of_two(bs, which):
    M, N, K = 300, 512, 1024
    A, sA, B, sB = _problem(M, N, K, seed=15, pow2=True)
    if which == "sA":
        sA[137, 9] = 0.75
    else:
        sB[5, 30] = 3.0
    _run_native(bs, A, sA, B, sB, M, N, K)
    assert bs.fp8_status_query() == bs._abi.FP8_ERR_SCALE
    assert bs.fp8_status_query() == 0   # the query clears the word


def test_pertoken_native_scales_only_4_byte_aligned(bs):
    """sA and sB need only 4-byte alignment: scales starting 4 bytes into an
    allocation give the same result as aligned copies, bit for bit."""
    M, N, K = 300, 256, 1024
    A, sA, B, sB = _problem(M, N, K, seed=16, pow2=True)
    C_ref = _run_native(bs, A, sA, B, sB, M, N, K)
    dA, dB = A.to(DEV), B.to(DEV)
    bufA = torch.empty(sA.numel() + 1, dtype=torch.float32, device=DEV)
    bufB = torch.empty(sB.numel() + 1, dtype=torch.float32, device=DEV)
    sA_off = bufA[1:].view(sA.shape)
    sB_off = bufB[1:].view(sB.shape)
    sA_off.copy_(sA.to(DEV))
    sB_off.copy_(sB.to(DEV))
    assert sA_off.data_ptr() % 16 == 4 and sB_off.data_ptr() % 16 == 4
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    bs.fp8_gemm_pertoken(dA, sA_off, dB, sB_off, C, M, N, K, mode=bs.FP8_PATH_NATIVE)
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == 0
    assert torch.equal(C.view(torch.int16), C_ref.view(torch.int16))


def test_pertoken_native_square_4096_rows(bs):
    """The bench's p1n shape (256 tiles on 76 CTA pairs, each pair running
    several tiles, so the per-row scale pipeline crosses tile boundaries):
    whole rows at tile edges and 60 random rows against the oracle."""
    M = N = K = 4096
    g = torch.Generator(device=DEV).manual_seed(9)
    A = workloads.normal_codes(M, K, g, DEV)
    B = workloads.normal_codes(N, K, g, DEV)
    sA = torch.ldexp(torch.ones(M, K // 32, device=DEV),
                     torch.randint(-4, 5, (M, K // 32), generator=g, device=DEV)).float()
    sB = workloads.pow2_scales(N, K // 32, -4, 4, g, DEV)
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    bs.fp8_gemm_pertoken(A, sA, B, sB, C, M, N, K, mode=bs.FP8_PATH_NATIVE)
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == 0
    rng = np.random.default_rng(9)
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, 2049, M - 1], rng.integers(0, M, 60)]))
    Ah, sAh, Bh, sBh = (t.cpu().numpy() for t in (A, sA, B, sB))
    Cr, T = oracle.gemm_pertoken(Ah[rows], sAh[rows], Bh, sBh, len(rows), N, K)   # whole rows
    Cg = C[torch.from_numpy(rows).to(DEV)]
    check(bf16_to_f64(Cg), Cr, T, "pertoken native 4096^3 rows")


# ------------------------------------------------- UE8M0 per-token scales
# fp8_gemm_pertoken_e8m0: sA as UE8M0 bytes (value 2^(e-127)); the oracle
# takes the same scales as fp32 powers of two.

def _e8_problem(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    A = workloads.normal_codes(M, K, g, "cpu")
    B = workloads.normal_codes(N, K, g, "cpu")
    e = torch.randint(127 - 6, 127 + 7, (M, K // 32), generator=g).to(torch.uint8)
    sA_f32 = torch.ldexp(torch.ones(M, K // 32), e.to(torch.int32) - 127).float()
    sB = workloads.pow2_scales(N, K // 32, -4, 4, g, "cpu")
    return A, e.contiguous(), sA_f32.contiguous(), B, sB.contiguous()


def _run_e8(bs, A, e, B, sB, M, N, K):
    buf = torch.full((M + 2, N), -7.0, dtype=torch.bfloat16, device=DEV)
    C = buf[1:M + 1]
    bs.fp8_gemm_pertoken_e8m0(A.to(DEV), e.to(DEV) if e.device.type == "cpu" else e, B.to(DEV), sB.to(DEV),
                              C, M, N, K)
    torch.cuda.synchronize()
    assert torch.all(buf[0] == -7.0) and torch.all(buf[-1] == -7.0), "store outside C"
    return C


@pytest.mark.parametrize("M,N,K", [(1, 256, 256), (77, 256, 160), (256, 512, 1024), (300, 288, 2048),
                                   (1000, 768, 1056)])
def test_pertoken_e8m0_parity_and_equals_fp32_native(bs, M, N, K):
    """Against the oracle with the scales as fp32 powers of two, and bit for
    bit against fp8_gemm_pertoken's native path given those fp32 scales.  K=160
    and 1056 are not multiples of 256 (bytes read one at a time)."""
    A, e, sA32, B, sB = _e8_problem(M, N, K, seed=3 * M + N + K)
    C = _run_e8(bs, A, e, B, sB, M, N, K)
    assert bs.fp8_status_query() == 0
    Cr, T = oracle.gemm_pertoken(A.numpy(), sA32.numpy(), B.numpy(), sB.numpy(), M, N, K)
    check(bf16_to_f64(C), Cr, T, f"pertoken e8m0 {M}x{N}x{K}")
    C32 = _run_native(bs, A, sA32, B, sB, M, N, K)
    assert bs.fp8_status_query() == 0
    assert torch.equal(C.view(torch.int16), C32.view(torch.int16))


def test_pertoken_e8m0_unaligned_bytes(bs):
    """sA starting one byte into an allocation (read byte by byte) gives the
    same bits as an aligned copy (read 8 bytes at a time)."""
    M, N, K = 300, 256, 2048
    A, e, _, B, sB = _e8_problem(M, N, K, seed=21)
    C_ref = _run_e8(bs, A, e, B, sB, M, N, K)
    buf = torch.empty(e.numel() + 1, dtype=torch.uint8, device=DEV)
    e_off = buf[1:].view(e.shape)
    e_off.copy_(e.to(DEV))
    assert e_off.data_ptr() % 8 == 1
    C = _run_e8(bs, A, e_off, B, sB, M, N, K)
    assert bs.fp8_status_query() == 0
    assert torch.equal(C.view(torch.int16), C_ref.view(torch.int16))


def test_pertoken_e8m0_reports_nan_byte(bs):
    M, N, K = 300, 512, 1024
    A, e, _, B, sB = _e8_problem(M, N, K, seed=22)
    e[211, 17] = 0xFF
    _run_e8(bs, A, e, B, sB, M, N, K)
    assert bs.fp8_status_query() == bs._abi.FP8_ERR_SCALE
    assert bs.fp8_status_query() == 0


def test_pertoken_e8m0_square_4096_rows(bs):
    """4096^3 (several tiles per CTA pair, the byte pipeline crossing tile
    boundaries, four entries in flight): whole rows against the oracle."""
    M = N = K = 4096
    A, e, sA32, B, sB = _e8_problem(M, N, K, seed=23)
    C = _run_e8(bs, A, e, B, sB, M, N, K)
    assert bs.fp8_status_query() == 0
    rng = np.random.default_rng(23)
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, 2049, M - 1], rng.integers(0, M, 40)]))
    Cr, T = oracle.gemm_pertoken(A.numpy()[rows], sA32.numpy()[rows], B.numpy(), sB.numpy(), len(rows), N, K)
    Cg = C[torch.from_numpy(rows).to(DEV)]
    check(bf16_to_f64(Cg), Cr, T, "pertoken e8m0 4096^3 rows")
