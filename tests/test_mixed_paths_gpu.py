"""Native and promotion tiles in one launch.

The path is chosen per output tile (all of a tile's block scales positive
normal powers of two: the block-scaled MMA; otherwise the exact fp32
promotion), and the two paths share the tensor memory of a CTA, so a CTA that
runs several tiles switches between them.  These problems have more tiles
than CTAs and a seeded mix of tile paths; every result is compared with the
oracle, and each tile must equal, bit for bit, the launch that forces its path
on the whole problem (FP8 GEMM library article, hncyxsy.com/news/241433,
section 3: the per-block scale decides how the block's partial sum is
promoted)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._accept import bf16_to_f64, check

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TILE = 256   # output tile of the single-problem kernel (CTA pair): 256 x 256


@pytest.fixture(scope="module")
def bs():
    import block_scaled_fp8_sm_gb300 as mod
    from block_scaled_fp8_sm_gb300 import build
    build.build()
    mod.library()
    return mod


def _mixed_problem(M, N, K, seed):
    """Power-of-two scales everywhere except one block in each selected
    256-row (sA) or 256-column (sB) band, which gets a factor 1.3."""
    g = torch.Generator().manual_seed(seed)
    A = workloads.normal_codes(M, K, g, "cpu")
    B = workloads.normal_codes(N, K, g, "cpu")
    sA = workloads.pow2_scales(M, K // 32, -3, 3, g, "cpu")
    sB = workloads.pow2_scales(N, K // 32, -3, 3, g, "cpu")
    mt, nt = (M + TILE - 1) // TILE, (N + TILE - 1) // TILE
    bad_m = torch.rand(mt, generator=g) < 0.3
    bad_n = torch.rand(nt, generator=g) < 0.2
    for t in range(mt):
        if bad_m[t]:
            rb = min(t * TILE // 32 + int(torch.randint(0, TILE // 32, (1,), generator=g)), sA.shape[0] - 1)
            sA[rb, int(torch.randint(0, K // 32, (1,), generator=g))] *= 1.3
    for t in range(nt):
        if bad_n[t]:
            cb = min(t * TILE // 32 + int(torch.randint(0, TILE // 32, (1,), generator=g)), sB.shape[0] - 1)
            sB[cb, int(torch.randint(0, K // 32, (1,), generator=g))] *= 1.3
    promote = bad_m[:, None] | bad_n[None, :]   # [mt, nt] tile path
    return workloads.Problem(A, sA, B, sB, M, N, K, name=f"mixed{M}x{N}x{K}"), promote


def _launch(bs, p, mode=None):
    A, sA, B, sB = (t.to(DEV) for t in (p.A, p.sA, p.B, p.sB))
    C = torch.full((p.M, p.N), -7.0, dtype=torch.bfloat16, device=DEV)
    bs.fp8_gemm_blockscaled(A, sA, B, sB, C, p.M, p.N, p.K, mode=mode)
    torch.cuda.synchronize()
    return C


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 160), (2304, 3328, 1056)])
def test_mixed_tiles_single_problem(bs, M, N, K):
    p, promote = _mixed_problem(M, N, K, seed=M + K)
    assert promote.any() and not promote.all()
    C = _launch(bs, p)
    assert bs.fp8_status_query() == 0

    # oracle on sampled elements (about 40 per tile) and whole rows at tile edges
    rng = np.random.default_rng(1)
    rows = [0, TILE - 1, TILE, M // 2 + 7, M - 1]
    ms = np.concatenate([rng.integers(0, M, 12000)] + [np.full(N, r) for r in rows])
    ns = np.concatenate([rng.integers(0, N, 12000)] + [np.arange(N) for _ in rows])
    Cr, T = oracle.gemm_sampled(p.A.numpy(), p.sA.numpy(), p.B.numpy(), p.sB.numpy(), M, N, K, ms, ns)
    Cg = C[torch.from_numpy(ms).to(DEV), torch.from_numpy(ns).to(DEV)]
    check(bf16_to_f64(Cg), Cr, T, p.name)

    # each tile equals the launch that forces its path everywhere
    Cp = _launch(bs, p, mode=2)
    Cn = _launch(bs, p, mode=1)
    assert bs.fp8_status_query() == bs._abi.FP8_ERR_SCALE   # forced native met the 1.3 blocks
    assert bs.fp8_status_query() == 0
    bits, bp, bn = (x.view(torch.int16) for x in (C, Cp, Cn))
    for mt in range(promote.shape[0]):
        for nt in range(promote.shape[1]):
            r = slice(mt * TILE, min(M, (mt + 1) * TILE))
            c = slice(nt * TILE, min(N, (nt + 1) * TILE))
            ref = bp if promote[mt, nt] else bn
            assert torch.equal(bits[r, c], ref[r, c]), f"tile ({mt},{nt}) promote={bool(promote[mt, nt])}"


def test_mixed_groups_grouped_kernel(bs):
    """Groups alternate between power-of-two and arbitrary scales; the
    launch has more 64-row tiles than SMs."""
    gp = workloads.grouped(seed=11, G=8, N=2048, K=256, Ms=[300, 17, 256, 64, 129, 1, 333, 200])
    g = torch.Generator().manual_seed(12)
    for i in range(0, gp.G, 2):
        gp.sA[i] = gp.sA[i] * (torch.rand(gp.sA[i].shape, generator=g) * 0.5 + 0.75)
    dev_A = gp.A.to(DEV)
    groups, outs = [], []
    for i in range(gp.G):
        o = gp.offsets[i]
        Cg = torch.full((gp.Ms[i] + 1, gp.N), -7.0, dtype=torch.bfloat16, device=DEV)
        outs.append(Cg)
        groups.append((dev_A[o:o + gp.Ms[i]], gp.sA[i].to(DEV), gp.B[i].to(DEV), gp.sB[i].to(DEV), Cg))
    Ms = torch.tensor(gp.Ms, dtype=torch.int32, device=DEV)
    bs.fp8_gemm_grouped(groups, Ms, gp.N, gp.K)
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == 0
    for i in range(gp.G):
        assert torch.all(outs[i][gp.Ms[i]:] == -7.0), f"group {i}: store past M_g"
        Cr, T = oracle.gemm(gp.A_group(i).numpy(), gp.sA[i].numpy(), gp.B[i].numpy(),
                            gp.sB[i].numpy(), gp.Ms[i], gp.N, gp.K)
        check(bf16_to_f64(outs[i][:gp.Ms[i]]), Cr, T, f"mixed group {i}")
