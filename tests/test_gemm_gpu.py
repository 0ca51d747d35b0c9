"""GPU parity of the block-scaled GEMM (called through the C ABI) against the
CPU oracle, element by element, on seeded inputs.

Small and ragged shapes are compared in full; the full-size workloads are
compared on sampled elements and whole sampled rows, in the same launch
configuration the benchmark times.  Tolerance: tests/_accept.py.
"""
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


def _to_dev(p):
    return (p.A.to(DEV), p.sA.to(DEV), p.B.to(DEV), p.sB.to(DEV))


def _run(bs, p, mode=None, guard=False):
    A, sA, B, sB = _to_dev(p)
    if guard:
        # sentinel rows before and after C catch stray stores
        buf = torch.full((p.M + 2, p.N), -7.0, dtype=torch.bfloat16, device=DEV)
        C = buf[1:p.M + 1]
    else:
        C = torch.empty(p.M, p.N, dtype=torch.bfloat16, device=DEV)
    bs.fp8_gemm_blockscaled(A, sA, B, sB, C, p.M, p.N, p.K, mode=mode)
    torch.cuda.synchronize()
    if guard:
        assert torch.all(buf[0] == -7.0) and torch.all(buf[-1] == -7.0), "store outside C"
    return C


def _full_check(bs, p, mode=None, what=""):
    C = _run(bs, p, mode=mode, guard=True)
    Cr, T = oracle.gemm(p.A.numpy(), p.sA.numpy(), p.B.numpy(), p.sB.numpy(), p.M, p.N, p.K)
    return check(bf16_to_f64(C), Cr, T, what or p.name)


def _rand_problem(M, N, K, seed, pow2=True, elo=-4, ehi=4):
    g = torch.Generator().manual_seed(seed)
    A = workloads.normal_codes(M, K, g, "cpu")
    B = workloads.normal_codes(N, K, g, "cpu")
    if pow2:
        sA = workloads.pow2_scales(M, K // 32, elo, ehi, g, "cpu")
        sB = workloads.pow2_scales(N, K // 32, elo, ehi, g, "cpu")
    else:
        sA = torch.rand((M + 31) // 32, K // 32, generator=g) * 2 + 0.05
        sB = torch.rand((N + 31) // 32, K // 32, generator=g) * 2 + 0.05
    return workloads.Problem(A, sA, B, sB, M, N, K, name=f"rand{M}x{N}x{K}{'' if pow2 else 'arb'}")


# ------------------------------------------------------------ small / ragged

def test_square256_native(bs):
    _full_check(bs, workloads.make("c0"))
    assert bs.fp8_status_query() == 0


@pytest.mark.parametrize("M,N,K", [(1, 32, 32), (7, 96, 160), (100, 160, 416), (129, 288, 96),
                                   (300, 256, 1056), (64, 32, 4096), (257, 384, 128)])
def test_ragged_native(bs, M, N, K):
    _full_check(bs, _rand_problem(M, N, K, seed=M + N + K))


@pytest.mark.parametrize("pow2", [True, False])
def test_multi_tile_partial_last_stage(bs, pow2):
    """4096 x 2560 x 1056: 160 pair tiles on 76 pairs (every pair runs two or
    three tiles) whose K loop ends in a partial 256-K stage (1056 = 4 x 256 +
    32): the full-stage straight line and the guarded stage body alternate
    within each tile, on both paths.  Compared in full."""
    _full_check(bs, _rand_problem(4096, 2560, 1056, seed=77 + pow2, pow2=pow2))
    assert bs.fp8_status_query() == 0


@pytest.mark.parametrize("M,N,K", [(1, 32, 32), (45, 96, 160), (130, 288, 480), (256, 256, 1024)])
def test_ragged_promote_arbitrary_scales(bs, M, N, K):
    _full_check(bs, _rand_problem(M, N, K, seed=M * 3 + K, pow2=False))


def test_outlier_small_promote(bs):
    _full_check(bs, workloads.outlier(n=512, seed=3))


@pytest.mark.parametrize("mode", [1, 2])
def test_forced_paths_on_power_of_two_scales(bs, mode):
    p = _rand_problem(200, 160, 352, seed=5)
    _full_check(bs, p, mode=mode, what=f"mode{mode}")
    assert bs.fp8_status_query() == 0


def test_forced_native_with_arbitrary_scales_reports_and_stays_correct(bs):
    p = _rand_problem(150, 96, 256, seed=6, pow2=False)
    _full_check(bs, p, mode=1, what="native-forced-arbitrary")
    assert bs.fp8_status_query() == bs._abi.FP8_ERR_SCALE
    assert bs.fp8_status_query() == 0


def test_k_zero_gives_zeros(bs):
    C = torch.full((40, 64), 3.0, dtype=torch.bfloat16, device=DEV)
    e = torch.empty(0, dtype=torch.uint8, device=DEV)
    f = torch.empty(0, dtype=torch.float32, device=DEV)
    bs.fp8_gemm_blockscaled(e, f, e, f, C, 40, 64, 0)
    torch.cuda.synchronize()
    assert torch.all(C == 0)


def test_run_to_run_bit_identical(bs):
    p = workloads.square(n=512, seed=9)
    c1 = _run(bs, p)
    c2 = _run(bs, p)
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


# --------------------------------------------------------------- full sizes

def _sampled_check(bs, p, C, n_samples=4000, rows=(0, 1), seed=0):
    """Compare random elements and whole rows of C with the oracle."""
    rng = np.random.default_rng(seed)
    ms = rng.integers(0, p.M, n_samples)
    ns = rng.integers(0, p.N, n_samples)
    row_list = [r for r in rows if r < p.M] + [p.M - 1]
    ms = np.concatenate([ms] + [np.full(p.N, r) for r in row_list])
    ns = np.concatenate([ns] + [np.arange(p.N) for _ in row_list])
    A, sA, B, sB = (t.cpu().numpy() for t in (p.A, p.sA, p.B, p.sB))
    Cr, T = oracle.gemm_sampled(A, sA, B, sB, p.M, p.N, p.K, ms, ns)
    Cg = C[torch.from_numpy(ms).to(C.device), torch.from_numpy(ns).to(C.device)]
    return check(bf16_to_f64(Cg), Cr, T, p.name)


@pytest.mark.parametrize("name", ["c1", "c4"])
def test_full_size_sampled(bs, name):
    p = workloads.make(name, seed=0, device=DEV)
    A, sA, B, sB = p.A, p.sA, p.B, p.sB
    C = torch.empty(p.M, p.N, dtype=torch.bfloat16, device=DEV)
    bs.fp8_gemm_blockscaled(A, sA, B, sB, C, p.M, p.N, p.K)
    torch.cuda.synchronize()
    _sampled_check(bs, p, C, rows=(0, 1, 127, 128, p.M // 2))
    assert bs.fp8_status_query() == 0


def test_prefill_size_sampled(bs):
    p = workloads.make("c2", seed=0, device=DEV)
    C = torch.empty(p.M, p.N, dtype=torch.bfloat16, device=DEV)
    bs.fp8_gemm_blockscaled(p.A, p.sA, p.B, p.sB, C, p.M, p.N, p.K)
    torch.cuda.synchronize()
    _sampled_check(bs, p, C, n_samples=3000, rows=(0, 4095))
    assert bs.fp8_status_query() == 0


# -------------------------------------------------------- batch invariance

@pytest.mark.parametrize("name,sizes", [("c4", (1, 7, 64, 8192)), ("c1", (1, 7, 64, 4096))])
def test_batch_invariance_bit_exact(bs, name, sizes):
    """The first 64 rows computed within launches of different M are
    bit-identical (the launch with M=1 gives row 0 only)."""
    p = workloads.make(name, seed=0, device=DEV)
    rows = {}
    for m in sizes:
        q = workloads.prefix_rows(p, m)
        C = torch.empty(m, p.N, dtype=torch.bfloat16, device=DEV)
        bs.fp8_gemm_blockscaled(q.A, q.sA, q.B, q.sB, C, m, p.N, p.K)
        torch.cuda.synchronize()
        rows[m] = C[:64].view(torch.int16).clone()
    ref = rows[max(sizes)]
    for m in sizes:
        k = min(m, 64)
        assert torch.equal(rows[m][:k], ref[:k]), f"M={m} differs"


def test_batch_invariance_pinned_promotion(bs):
    """With the promotion path pinned (single-CTA tiles), the first rows are
    bit-identical across launches of different M, and equal to what AUTO
    computes for them when their tile promotes (the 8192^3 outlier data)."""
    p = workloads.make("c4", seed=0, device=DEV)
    N, K = 512, 2048   # a slice of the outlier problem: B rows and K columns prefixes
    B = p.B[:N, :K].contiguous()
    sB = p.sB[:N // 32, :K // 32].contiguous()
    rows = {}
    for m in (1, 7, 64, 300):
        A = p.A[:m, :K].contiguous()
        sA = p.sA[:(m + 31) // 32, :K // 32].contiguous()
        C = torch.empty(m, N, dtype=torch.bfloat16, device=DEV)
        bs.fp8_gemm_blockscaled(A, sA, B, sB, C, m, N, K, mode=2)
        torch.cuda.synchronize()
        rows[m] = C[:64].view(torch.int16).clone()
        if m == 300:
            Ca = torch.empty(m, N, dtype=torch.bfloat16, device=DEV)
            bs.fp8_gemm_blockscaled(A, sA, B, sB, Ca, m, N, K)
            torch.cuda.synchronize()
            assert torch.equal(Ca.view(torch.int16), C.view(torch.int16)), "AUTO vs pinned promotion"
    for m in (1, 7, 64):
        k = min(m, 64)
        assert torch.equal(rows[m][:k], rows[300][:k]), f"M={m} differs"
    assert bs.fp8_status_query() == 0


# ------------------------------------------------------------------- grouped

def _grouped_run(bs, gp, mode=None):
    dev_A = gp.A.to(DEV)
    groups, outs = [], []
    for g in range(gp.G):
        o = gp.offsets[g]
        Cg = torch.full((max(gp.Ms[g], 1) + 1, gp.N), -7.0, dtype=torch.bfloat16, device=DEV)
        outs.append(Cg)
        groups.append((dev_A[o:o + gp.Ms[g]] if gp.Ms[g] else dev_A, gp.sA[g].to(DEV) if gp.sA[g].numel() else gp.sB[g].to(DEV),
                       gp.B[g].to(DEV), gp.sB[g].to(DEV), Cg))
    Ms = torch.tensor(gp.Ms, dtype=torch.int32, device=DEV)
    bs.fp8_gemm_grouped(groups, Ms, gp.N, gp.K, mode=mode)
    torch.cuda.synchronize()
    for g in range(gp.G):
        assert torch.all(outs[g][gp.Ms[g]:] == -7.0), f"group {g}: store past M_g"
    return [outs[g][:gp.Ms[g]] for g in range(gp.G)], groups


def test_grouped_small_full(bs):
    gp = workloads.grouped(seed=1, G=6, N=288, K=416, Ms=[0, 1, 33, 130, 64, 200])
    outs, _ = _grouped_run(bs, gp)
    for g in range(gp.G):
        if gp.Ms[g] == 0:
            continue
        Cr, T = oracle.gemm(gp.A_group(g).numpy(), gp.sA[g].numpy(), gp.B[g].numpy(),
                            gp.sB[g].numpy(), gp.Ms[g], gp.N, gp.K)
        check(bf16_to_f64(outs[g]), Cr, T, f"group{g}")
    assert bs.fp8_status_query() == 0


def test_grouped_equals_plain_bit_exact(bs):
    gp = workloads.grouped(seed=2, G=5, N=256, K=512, Ms=[3, 64, 1, 129, 40])
    outs, groups = _grouped_run(bs, gp)
    for g in range(gp.G):
        A, sA, B, sB, _ = groups[g]
        C = torch.empty(gp.Ms[g], gp.N, dtype=torch.bfloat16, device=DEV)
        bs.fp8_gemm_blockscaled(A, sA, B, sB, C, gp.Ms[g], gp.N, gp.K)
        torch.cuda.synchronize()
        assert torch.equal(C.view(torch.int16), outs[g].view(torch.int16)), f"group {g}"


def test_grouped_decode_size_sampled(bs):
    gp = workloads.make("c3", seed=0, device=DEV)
    outs, _ = _grouped_run(bs, gp)
    rng = np.random.default_rng(0)
    A = gp.A.cpu().numpy()
    for g in range(gp.G):
        Mg = gp.Ms[g]
        ms = np.concatenate([rng.integers(0, Mg, 300), np.full(gp.N, Mg - 1)])
        ns = np.concatenate([rng.integers(0, gp.N, 300), np.arange(gp.N)])
        o = gp.offsets[g]
        Cr, T = oracle.gemm_sampled(A[o:o + Mg], gp.sA[g].cpu().numpy(), gp.B[g].cpu().numpy(),
                                    gp.sB[g].cpu().numpy(), Mg, gp.N, gp.K, ms, ns)
        Cg = outs[g][torch.from_numpy(ms).to(DEV), torch.from_numpy(ns).to(DEV)]
        check(bf16_to_f64(Cg), Cr, T, f"c3 group {g}")
    assert bs.fp8_status_query() == 0


def test_grouped_arbitrary_scales_promote(bs):
    g = torch.Generator().manual_seed(4)
    gp = workloads.grouped(seed=4, G=3, N=96, K=256, Ms=[5, 70, 129])
    gp.sA = [torch.rand(s.shape, generator=g) + 0.1 for s in gp.sA]
    gp.sB = [torch.rand(s.shape, generator=g) + 0.1 for s in gp.sB]
    outs, _ = _grouped_run(bs, gp)
    for i in range(gp.G):
        Cr, T = oracle.gemm(gp.A_group(i).numpy(), gp.sA[i].numpy(), gp.B[i].numpy(),
                            gp.sB[i].numpy(), gp.Ms[i], gp.N, gp.K)
        check(bf16_to_f64(outs[i]), Cr, T, f"group{i}")


def test_grouped_prebuilt_descriptors_same_bits(bs):
    gp = workloads.grouped(seed=3, G=4, N=160, K=224, Ms=[9, 64, 1, 30])
    outs, groups = _grouped_run(bs, gp)
    again = [torch.empty_like(o) for o in outs]
    descs = bs.group_descs([(a, sa, b, sb, c) for (a, sa, b, sb, _), c in zip(groups, again)])
    Ms = torch.tensor(gp.Ms, dtype=torch.int32, device=DEV)
    for _ in range(2):   # the same descriptor array serves repeated calls
        bs.fp8_gemm_grouped(descs, Ms, gp.N, gp.K)
    torch.cuda.synchronize()
    for g in range(gp.G):
        assert torch.equal(again[g].view(torch.int16), outs[g].view(torch.int16)), f"group {g}"
