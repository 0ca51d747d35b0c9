"""A seeded sweep of random problem shapes through every GEMM entry point of the
C ABI, against the oracle: M from 1 to 300, N and K multiples of 32 from 32 to
512 (one-block N and K, K ending inside a 128-K stage, M ending inside a
32-row block, tiles cut at every edge).  Per shape: the block-scaled call in
each path mode, the allocation-free call, the quantized-output call, the
residual, per-token x per-channel and per-token calls, and a two-group grouped
launch; the allocation-free call, the pinned promotion path and the
quantized-output call are also compared with the regular call (followed by
the block quantizer) bit for bit where their contracts say they agree."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._accept import bf16_to_f64, check

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
CASES = 24


@pytest.fixture(scope="module")
def bs():
    import block_scaled_fp8_sm_gb300 as mod
    from block_scaled_fp8_sm_gb300 import build
    build.build()
    mod.library()
    return mod


def _shape(i):
    rng = np.random.default_rng(1000 + i)
    M = int(rng.integers(1, 301))
    N = 32 * int(rng.integers(1, 17))
    K = 32 * int(rng.integers(1, 17))
    return M, N, K


@pytest.mark.parametrize("i", range(CASES))
def test_random_shape_every_entry_point(bs, i):
    M, N, K = _shape(i)
    g = torch.Generator().manual_seed(2000 + i)
    A = workloads.normal_codes(M, K, g, "cpu")
    B = workloads.normal_codes(N, K, g, "cpu")
    sA_p = workloads.pow2_scales(M, K // 32, -4, 4, g, "cpu")
    sB_p = workloads.pow2_scales(N, K // 32, -4, 4, g, "cpu")
    sA_a = torch.rand((M + 31) // 32, K // 32, generator=g) * 2 + 0.05
    sB_a = torch.rand(N // 32, K // 32, generator=g) * 2 + 0.05
    dA, dB = A.to(DEV), B.to(DEV)
    Ah, Bh = A.numpy(), B.numpy()
    tag = f"random {M}x{N}x{K}"

    def out():
        return torch.empty(M, N, dtype=torch.bfloat16, device=DEV)

    # block scales: power-of-two (AUTO, NATIVE), arbitrary (AUTO, PROMOTE)
    for kind, sA, sB in (("pow2", sA_p, sB_p), ("arb", sA_a, sB_a)):
        Cr, T = oracle.gemm(Ah, sA.numpy(), Bh, sB.numpy(), M, N, K)
        modes = (None, bs.FP8_PATH_NATIVE) if kind == "pow2" else (None, bs.FP8_PATH_PROMOTE)
        res = {}
        for mode in modes:
            C = out()
            bs.fp8_gemm_blockscaled(dA, sA.to(DEV), dB, sB.to(DEV), C, M, N, K, mode=mode)
            torch.cuda.synchronize()
            assert bs.fp8_status_query() == 0
            check(bf16_to_f64(C), Cr, T, f"{tag} {kind} mode {mode}")
            res[mode] = C
        if kind == "arb":
            # AUTO promotes every tile here; its promoted tiles equal PROMOTE's bits
            assert torch.equal(res[None].view(torch.int16), res[bs.FP8_PATH_PROMOTE].view(torch.int16))
        # the allocation-free call: same bits as the regular call on single-kind scales
        C = out()
        bs.fp8_gemm_blockscaled_noalloc(dA, sA.to(DEV), dB, sB.to(DEV), C, M, N, K)
        torch.cuda.synchronize()
        assert bs.fp8_status_query() == 0
        assert torch.equal(C.view(torch.int16), res[None].view(torch.int16))

    # output quantized in the epilogue: the bf16 call followed by the quantizer, bit for bit
    for sA, sB in ((sA_p, sB_p), (sA_a, sB_a)):
        C = out()
        bs.fp8_gemm_blockscaled(dA, sA.to(DEV), dB, sB.to(DEV), C, M, N, K)
        q_ref, s_ref = bs.fp8_quantize_blocks(C)
        Cq = torch.empty(M, N, dtype=torch.uint8, device=DEV)
        sC = torch.empty((M + 31) // 32, N // 32, dtype=torch.float32, device=DEV)
        bs.fp8_gemm_blockscaled_quant(dA, sA.to(DEV), dB, sB.to(DEV), Cq, sC, M, N, K)
        torch.cuda.synchronize()
        assert bs.fp8_status_query() == 0
        assert torch.equal(Cq, q_ref) and torch.equal(sC.view(torch.int32), s_ref.view(torch.int32)), f"{tag} quant"

    # residual (in place)
    gr = torch.Generator().manual_seed(3000 + i)
    R = torch.randn(M, N, generator=gr).to(torch.bfloat16)
    C = R.to(DEV).clone()
    bs.fp8_gemm_blockscaled_residual(dA, sA_p.to(DEV), dB, sB_p.to(DEV), C, C, M, N, K)
    torch.cuda.synchronize()
    Cr, T = oracle.gemm_residual(Ah, sA_p.numpy(), Bh, sB_p.numpy(), R.view(torch.int16).numpy(), M, N, K)
    check(bf16_to_f64(C), Cr, T, f"{tag} residual in place")

    # per-token x per-channel
    sr = torch.rand(M, generator=g) + 0.5
    sc = torch.rand(N, generator=g) + 0.5
    C = out()
    bs.fp8_gemm_rowcol(dA, sr.to(DEV), dB, sc.to(DEV), C, M, N, K)
    torch.cuda.synchronize()
    Cr, T = oracle.gemm_rowcol(Ah, sr.numpy(), Bh, sc.numpy(), M, N, K)
    check(bf16_to_f64(C), Cr, T, f"{tag} rowcol")

    # per-token 1x32 A scales: arbitrary (promotion) and powers of two (native)
    sT_a = torch.rand(M, K // 32, generator=g) * 2 + 0.05
    sT_p = torch.ldexp(torch.ones(M, K // 32), torch.randint(-4, 5, (M, K // 32), generator=g)).float()
    for kind, sT, sB, mode in (("arb", sT_a, sB_a, None), ("pow2", sT_p, sB_p, bs.FP8_PATH_NATIVE)):
        C = out()
        bs.fp8_gemm_pertoken(dA, sT.to(DEV), dB, sB.to(DEV), C, M, N, K, mode=mode)
        torch.cuda.synchronize()
        assert bs.fp8_status_query() == 0
        Cr, T = oracle.gemm_pertoken(Ah, sT.numpy(), Bh, sB.numpy(), M, N, K)
        check(bf16_to_f64(C), Cr, T, f"{tag} pertoken {kind}")

    # grouped: the same problem split into two groups at a ragged row
    cut = M // 3
    Ms = [cut, M - cut]
    offs = [0, cut]
    sA_g = [workloads.pow2_scales(m, K // 32, -4, 4, g, "cpu") for m in Ms]
    Cs = [torch.empty(max(m, 1), N, dtype=torch.bfloat16, device=DEV) for m in Ms]
    groups = [(dA[o:o + m] if m else dA[:1], s.to(DEV) if m else sA_p[:1].to(DEV), dB, sB_p.to(DEV), c)
              for o, m, s, c in zip(offs, Ms, sA_g, Cs)]
    bs.fp8_gemm_grouped(groups, torch.tensor(Ms, dtype=torch.int32, device=DEV), N, K)
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == 0
    for o, m, s, c in zip(offs, Ms, sA_g, Cs):
        if m == 0:
            continue
        Cr, T = oracle.gemm(Ah[o:o + m], s.numpy(), Bh, sB_p.numpy(), m, N, K)
        check(bf16_to_f64(c[:m]), Cr, T, f"{tag} grouped rows {o}..{o + m}")
