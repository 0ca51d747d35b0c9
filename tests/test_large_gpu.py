"""Outputs past 2^31 elements: the entry points take M, N, K up to 2^31 - 1
each, so output offsets need 64-bit arithmetic.  C here is 70000 x 32768
bf16 (2.29e9 elements, 4.6 GB): rows from 65536 on start beyond element
offset 2^31 and rows from 32768 on beyond byte offset 2^31.  K = 64 keeps the
work small.  M = 70000 ends inside a 256-row tile.

Checked: guard rows around C, the device status, and sampled elements plus
whole rows on both sides of each boundary against the oracle; the quantized
output (E4M3 codes, 2.29e9 bytes) against the GEMM followed by the block
quantizer, bit for bit over the whole arrays; the per-token x per-channel and
per-token (1 x 32 along K) scale forms on whole rows, whose oracle takes the
selected rows of A and of their scales; a grouped call whose first group has
70000 rows.  Tolerance: tests/_accept.py.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._accept import bf16_to_f64, check

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
M, N, K = 70000, 32768, 64
ROWS = (0, 32767, 32768, 65535, 65536, 65537, 69887, 69888, M - 1)


@pytest.fixture(scope="module")
def bs():
    import block_scaled_fp8_sm_gb300 as mod
    from block_scaled_fp8_sm_gb300 import build
    build.build()
    mod.library()
    return mod


def _problem(seed, pow2):
    g = torch.Generator().manual_seed(seed)
    A = workloads.normal_codes(M, K, g, "cpu")
    B = workloads.normal_codes(N, K, g, "cpu")
    if pow2:
        sA = workloads.pow2_scales(M, K // 32, -4, 4, g, "cpu")
        sB = workloads.pow2_scales(N, K // 32, -4, 4, g, "cpu")
    else:
        sA = torch.rand((M + 31) // 32, K // 32, generator=g) * 2 + 0.05
        sB = torch.rand(N // 32, K // 32, generator=g) * 2 + 0.05
    return A, sA, B, sB


def _sampled(A, sA, B, sB, C, seed):
    rng = np.random.default_rng(seed)
    ms = np.concatenate([rng.integers(0, M, 3000), rng.integers(65536, M, 3000)] +
                        [np.full(N, r) for r in ROWS])
    ns = np.concatenate([rng.integers(0, N, 6000)] + [np.arange(N) for _ in ROWS])
    Cr, T = oracle.gemm_sampled(A.numpy(), sA.numpy(), B.numpy(), sB.numpy(), M, N, K, ms, ns)
    Cg = C[torch.from_numpy(ms).to(DEV), torch.from_numpy(ns).to(DEV)]
    return Cg, Cr, T


@pytest.mark.parametrize("pow2,mode", [(True, None), (False, None), (False, 2)])
def test_output_past_2_31_elements(bs, pow2, mode):
    """AUTO on power-of-two scales (native tiles), AUTO on arbitrary scales
    (promotion tiles on CTA pairs), PROMOTE (the single-CTA kernel)."""
    A, sA, B, sB = _problem(seed=31 if pow2 else 32, pow2=pow2)
    buf = torch.full((M + 2, N), -7.0, dtype=torch.bfloat16, device=DEV)
    C = buf[1:M + 1]
    bs.fp8_gemm_blockscaled(A.to(DEV), sA.to(DEV), B.to(DEV), sB.to(DEV), C, M, N, K, mode=mode)
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == 0
    assert torch.all(buf[0] == -7.0) and torch.all(buf[-1] == -7.0), "store outside C"
    Cg, Cr, T = _sampled(A, sA, B, sB, C, seed=5)
    check(bf16_to_f64(Cg), Cr, T, f"70000x32768x64 {'pow2' if pow2 else 'arb'} mode {mode}")
    del buf, C
    torch.cuda.empty_cache()


def test_quantized_output_past_2_31_bytes(bs):
    A, sA, B, sB = (t.to(DEV) for t in _problem(seed=33, pow2=True))
    Cq = torch.empty(M, N, dtype=torch.uint8, device=DEV)
    sC = torch.empty((M + 31) // 32, N // 32, dtype=torch.float32, device=DEV)
    bs.fp8_gemm_blockscaled_quant(A, sA, B, sB, Cq, sC, M, N, K)
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    bs.fp8_gemm_blockscaled(A, sA, B, sB, C, M, N, K)
    q, s = bs.fp8_quantize_blocks(C)
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == 0
    assert torch.equal(Cq, q)
    assert torch.equal(sC.view(torch.int32), s.view(torch.int32))
    del Cq, sC, C, q, s
    torch.cuda.empty_cache()


def _guarded():
    buf = torch.full((M + 2, N), -7.0, dtype=torch.bfloat16, device=DEV)
    return buf, buf[1:M + 1]


def _rows_check(buf, C, Cr, T, what):
    assert torch.all(buf[0] == -7.0) and torch.all(buf[-1] == -7.0), "store outside C"
    rows = torch.tensor(ROWS, device=DEV)
    check(bf16_to_f64(C[rows]), Cr, T, what)


def test_rowcol_past_2_31_elements(bs):
    g = torch.Generator().manual_seed(34)
    A = workloads.normal_codes(M, K, g, "cpu")
    B = workloads.normal_codes(N, K, g, "cpu")
    sA = (torch.rand(M, generator=g) * 4 - 2).float()
    sB = (torch.rand(N, generator=g) * 3).float()
    buf, C = _guarded()
    bs.fp8_gemm_rowcol(A.to(DEV), sA.to(DEV), B.to(DEV), sB.to(DEV), C, M, N, K)
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == 0
    r = list(ROWS)
    Cr, T = oracle.gemm_rowcol(A.numpy()[r], sA.numpy()[r], B.numpy(), sB.numpy(), len(r), N, K)
    _rows_check(buf, C, Cr, T, "rowcol 70000x32768x64 rows")
    del buf, C
    torch.cuda.empty_cache()


@pytest.mark.parametrize("form", ["promote", "e8m0"])
def test_pertoken_past_2_31_elements(bs, form):
    """Arbitrary per-token scales (AUTO: the single-CTA promotion kernel) and
    UE8M0 bytes (the native CTA-pair kernel)."""
    g = torch.Generator().manual_seed(35)
    A = workloads.normal_codes(M, K, g, "cpu")
    B = workloads.normal_codes(N, K, g, "cpu")
    sB = workloads.pow2_scales(N, K // 32, -4, 4, g, "cpu")
    buf, C = _guarded()
    if form == "promote":
        sA = (torch.rand(M, K // 32, generator=g) * 2 + 0.05).float()
        bs.fp8_gemm_pertoken(A.to(DEV), sA.to(DEV), B.to(DEV), sB.to(DEV), C, M, N, K)
    else:
        e = torch.randint(127 - 6, 127 + 7, (M, K // 32), generator=g).to(torch.uint8)
        sA = torch.ldexp(torch.ones(M, K // 32), e.to(torch.int32) - 127).float()
        bs.fp8_gemm_pertoken_e8m0(A.to(DEV), e.to(DEV), B.to(DEV), sB.to(DEV), C, M, N, K)
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == 0
    r = list(ROWS)
    Cr, T = oracle.gemm_pertoken(A.numpy()[r], sA.numpy()[r], B.numpy(), sB.numpy(), len(r), N, K)
    _rows_check(buf, C, Cr, T, f"pertoken {form} 70000x32768x64 rows")
    del buf, C
    torch.cuda.empty_cache()


def test_grouped_past_2_31_elements(bs):
    """The grouped call (64-row tiles, 16-byte global stores) with one group
    of 70000 rows and one of 5."""
    Ms = [M, 5]
    g = torch.Generator().manual_seed(36)
    probs = []
    for Mg in Ms:
        A = workloads.normal_codes(Mg, K, g, "cpu")
        B = workloads.normal_codes(N, K, g, "cpu")
        sA = workloads.pow2_scales(Mg, K // 32, -4, 4, g, "cpu")
        sB = workloads.pow2_scales(N, K // 32, -4, 4, g, "cpu")
        probs.append((A, sA, B, sB))
    outs, groups = [], []
    for Mg, (A, sA, B, sB) in zip(Ms, probs):
        Cg = torch.full((Mg + 1, N), -7.0, dtype=torch.bfloat16, device=DEV)
        outs.append(Cg)
        groups.append((A.to(DEV), sA.to(DEV), B.to(DEV), sB.to(DEV), Cg))
    bs.fp8_gemm_grouped(groups, torch.tensor(Ms, dtype=torch.int32, device=DEV), N, K)
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == 0
    for Mg, Cg in zip(Ms, outs):
        assert torch.all(Cg[Mg] == -7.0), "store past M_g"
    A, sA, B, sB = probs[0]
    r = [x for x in ROWS]
    ms = np.concatenate([np.full(N, x) for x in r])
    ns = np.concatenate([np.arange(N) for _ in r])
    Cr, T = oracle.gemm_sampled(A.numpy(), sA.numpy(), B.numpy(), sB.numpy(), M, N, K, ms, ns)
    check(bf16_to_f64(outs[0][torch.tensor(r, device=DEV)].reshape(-1)), Cr, T, "grouped 70000x32768x64 rows")
    A, sA, B, sB = probs[1]
    Cr, T = oracle.gemm(A.numpy(), sA.numpy(), B.numpy(), sB.numpy(), 5, N, K)
    check(bf16_to_f64(outs[1][:5]), Cr, T, "grouped 5x32768x64")
    del outs, groups
    torch.cuda.empty_cache()
