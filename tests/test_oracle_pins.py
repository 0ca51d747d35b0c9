"""Pins for the CPU oracle: each check is fixed by something other than the
oracle itself (the format definition, the pages' rounding example, exact
rational arithmetic, identity / one-hot operands, closed forms, invariants).
A planted mistake in any part of the oracle's GEMM fails at least one of them
(see test_planted_mistakes_are_caught).  CPU only.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ------------------------------------------------------------------ E4M3 ----

def _e4m3_fraction(code):
    """Exact value of an E4M3 code from the bit fields (None for NaN)."""
    s, e, m = code >> 7, (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return None
    v = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -v if s else v


def test_e4m3_table_matches_bitfield_definition():
    tab = oracle.e4m3_table()
    for c in range(256):
        ref = _e4m3_fraction(c)
        if ref is None:
            assert math.isnan(tab[c]), hex(c)
        else:
            assert Fraction(tab[c]) == ref, hex(c)
            if ref == 0:
                assert math.copysign(1.0, tab[c]) == (-1.0 if c & 0x80 else 1.0)


def test_e4m3_table_matches_torch_cast():
    tab = oracle.e4m3_table()
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(tab)
    assert np.array_equal(nan, np.isnan(t))
    assert np.array_equal(tab[~nan], t[~nan])


def test_e4m3_named_values_golden():
    tab = oracle.e4m3_table()
    for code, val in _read_golden("e4m3_named_values.txt"):
        c = int(code, 16)
        if val == "nan":
            assert math.isnan(tab[c])
        else:
            assert tab[c] == float(val)
            assert math.copysign(1.0, tab[c]) == math.copysign(1.0, float(val))
    assert np.nanmax(tab) == 448.0


def test_e4m3_quantize_agrees_with_brute_force_and_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(4000) * 3, rng.standard_normal(2000) * 200,
                        rng.standard_normal(1000) * 1e-3, [0.0, -0.0, 448.0, -448.0]])
    x = x.astype(np.float32).astype(np.float64)
    q = oracle.e4m3_quantize(x)
    tab = oracle.e4m3_table()
    finite = np.array([c for c in range(256) if not math.isnan(tab[c])])
    # brute force nearest with ties to even code, saturating
    for xi, qi in zip(x[:500], q[:500]):
        a = min(abs(xi), 448.0)
        d = np.abs(np.abs(tab[finite]) - a)
        best = finite[(d == d.min())]
        best = [c & 0x7F for c in best]
        even = [c for c in best if c % 2 == 0]
        assert (qi & 0x7F) == (even[0] if even else best[0])
    # torch's own cast (an independent implementation of the same rounding)
    t = torch.from_numpy(np.clip(x, -448, 448).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, t)


def test_rounding_ties_golden():
    tab = oracle.e4m3_table()
    for fmt, inp, exp in _read_golden("rounding_ties.txt"):
        x, e = float(inp), float(exp)
        if fmt == "fp16":
            # the pages' own example; checked with numpy's IEEE half
            assert float(np.float16(x)) == e
        elif fmt == "bf16":
            bits = oracle.bf16_rne([x])[0]
            assert oracle.bf16_value([bits])[0] == e
        elif fmt == "e4m3":
            assert tab[oracle.e4m3_quantize([x])[0]] == e


def test_bf16_rne_matches_torch_cast():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        [0.0, -0.0, 1.0, 3.3895313892515355e38, 1e-40, -1e-42]])
    x32 = x.astype(np.float32)
    ours = oracle.bf16_rne(x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# ------------------------------------------------------------------ GEMM ----

def _rand_problem(M, N, K, seed, elo=-4, ehi=4, arbitrary=False):
    rng = np.random.default_rng(seed)
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    A = rng.choice(codes, size=(M, K))
    B = rng.choice(codes, size=(N, K))
    if arbitrary:
        sA = (rng.random(((M + 31) // 32, K // 32)) * 3 + 0.01).astype(np.float32)
        sB = (rng.random(((N + 31) // 32, K // 32)) * 3 + 0.01).astype(np.float32)
    else:
        sA = np.ldexp(1.0, rng.integers(elo, ehi + 1, ((M + 31) // 32, K // 32))).astype(np.float32)
        sB = np.ldexp(1.0, rng.integers(elo, ehi + 1, ((N + 31) // 32, K // 32))).astype(np.float32)
    return A, sA, B, sB


def _exact(A, sA, B, sB, M, N, K):
    """C and T as exact rationals, straight from the definition."""
    val = [_e4m3_fraction(c) for c in range(256)]
    C = [[None] * N for _ in range(M)]
    T = [[None] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            mag = Fraction(0)
            for kb in range(K // 32):
                s = sum((val[A[m, k]] * val[B[n, k]] for k in range(32 * kb, 32 * kb + 32)), Fraction(0))
                sabs = sum((abs(val[A[m, k]] * val[B[n, k]]) for k in range(32 * kb, 32 * kb + 32)), Fraction(0))
                sc = Fraction(float(sA[m // 32, kb])) * Fraction(float(sB[n // 32, kb]))
                acc += sc * s
                mag += abs(sc) * sabs
            C[m][n] = acc
            T[m][n] = mag
    return C, T


@pytest.mark.parametrize("M,N,K,elo,ehi", [(5, 7, 64, -1, 1), (33, 34, 96, -2, 2), (1, 40, 128, 0, 0)])
def test_brute_force_exact_small_exponent_range(M, N, K, elo, ehi):
    A, sA, B, sB = _rand_problem(M, N, K, seed=M * 100 + N, elo=elo, ehi=ehi)
    C, T = oracle.gemm(A, sA, B, sB, M, N, K, nthreads=2)
    Ce, Te = _exact(A, sA, B, sB, M, N, K)
    for m in range(M):
        for n in range(N):
            # with this exponent range every partial sum fits in 53 bits: exact
            assert Fraction(C[m, n]) == Ce[m][n]
            assert Fraction(T[m, n]) == Te[m][n]


@pytest.mark.parametrize("arbitrary", [False, True])
def test_brute_force_within_fp64_bound(arbitrary):
    M, N, K = 37, 33, 160
    A, sA, B, sB = _rand_problem(M, N, K, seed=7, elo=-8, ehi=8, arbitrary=arbitrary)
    C, T = oracle.gemm(A, sA, B, sB, M, N, K)
    Ce, Te = _exact(A, sA, B, sB, M, N, K)
    u = 2.0 ** -53
    for m in range(M):
        for n in range(N):
            # one rounding per scaled block plus one per addition: 2*KB ulps of T
            bound = 2 * (K // 32 + 1) * u * float(Te[m][n])
            assert abs(Fraction(C[m, n]) - Ce[m][n]) <= Fraction(bound)
            assert abs(Fraction(T[m, n]) - Te[m][n]) <= Fraction(bound)


def test_identity_weights_reproduce_activations():
    M, K = 70, 96
    N = K
    rng = np.random.default_rng(3)
    A, sA, _, _ = _rand_problem(M, N, K, seed=3)
    B = np.zeros((N, K), dtype=np.uint8)
    B[np.arange(N), np.arange(K)] = 0x38                      # 1.0
    sB = np.ldexp(1.0, rng.integers(-3, 4, (N // 32, K // 32))).astype(np.float32)
    C, _ = oracle.gemm(A, sA, B, sB, M, N, K)
    tab = oracle.e4m3_table()
    exp = np.empty((M, N))
    for m in range(M):
        for n in range(N):
            exp[m, n] = float(sA[m // 32, n // 32]) * float(sB[n // 32, n // 32]) * tab[A[m, n]]
    assert np.array_equal(C, exp)
    ones_a = np.ones_like(sA)
    ones_b = np.ones_like(sB)
    C1, _ = oracle.gemm(A, ones_a, B, ones_b, M, N, K)
    assert np.array_equal(C1, tab[A].astype(np.float64))


def test_one_hot_row_picks_weights():
    M, N, K = 32, 64, 128
    _, _, B, sB = _rand_problem(M, N, K, seed=4)
    tab = oracle.e4m3_table()
    A = np.zeros((M, K), dtype=np.uint8)
    ks = np.random.default_rng(4).integers(0, K, M)
    A[np.arange(M), ks] = 0x40                                   # 2.0
    sA = np.full((1, K // 32), 0.25, dtype=np.float32)
    C, _ = oracle.gemm(A, sA, B, sB, M, N, K)
    for m in range(M):
        k = ks[m]
        exp = 0.25 * 2.0 * sB[np.arange(N) // 32, k // 32].astype(np.float64) * tab[B[:, k]]
        assert np.array_equal(C[m], exp)


def test_per_tensor_scales_closed_form():
    M, N, K = 50, 64, 256
    A, _, B, _ = _rand_problem(M, N, K, seed=5)
    tab = oracle.e4m3_table()
    alpha, beta = 2.0 ** -3, 2.0 ** 5
    sA = np.full(((M + 31) // 32, K // 32), alpha, dtype=np.float32)
    sB = np.full((N // 32, K // 32), beta, dtype=np.float32)
    C, _ = oracle.gemm(A, sA, B, sB, M, N, K)
    # every partial sum is a multiple of 2^-18 below 2^35: the fp64 matmul is exact
    ref = alpha * beta * (tab[A] @ tab[B].T)
    assert np.array_equal(C, ref)


def test_per_channel_scales_closed_form():
    M, N, K = 64, 96, 128
    A, _, B, _ = _rand_problem(M, N, K, seed=6)
    tab = oracle.e4m3_table()
    rng = np.random.default_rng(6)
    a = np.ldexp(1.0, rng.integers(-4, 5, M // 32))
    b = np.ldexp(1.0, rng.integers(-4, 5, N // 32))
    sA = np.repeat(a[:, None], K // 32, axis=1).astype(np.float32)
    sB = np.repeat(b[:, None], K // 32, axis=1).astype(np.float32)
    C, _ = oracle.gemm(A, sA, B, sB, M, N, K)
    ref = (np.repeat(a, 32)[:, None] * (tab[A] @ tab[B].T)) * np.repeat(b, 32)[None, :]
    assert np.array_equal(C, ref)


def test_block_rescale_invariant():
    """Doubling one block's data and halving its scale leaves C unchanged."""
    M, N, K = 64, 64, 128
    rng = np.random.default_rng(8)
    tab = oracle.e4m3_table()
    small = np.array([c for c in range(256) if not math.isnan(tab[c]) and abs(tab[c]) <= 224], dtype=np.uint8)
    A = rng.choice(small, size=(M, K))
    B = rng.choice(small, size=(N, K))
    sA = (rng.random((M // 32, K // 32)) * 4 + 0.1).astype(np.float32)
    sB = (rng.random((N // 32, K // 32)) * 4 + 0.1).astype(np.float32)
    C0, T0 = oracle.gemm(A, sA, B, sB, M, N, K)
    for (mb, kb) in [(0, 0), (1, 3), (0, 2)]:
        A2 = A.copy()
        blk = tab[A2[mb * 32:(mb + 1) * 32, kb * 32:(kb + 1) * 32]] * 2.0
        A2[mb * 32:(mb + 1) * 32, kb * 32:(kb + 1) * 32] = oracle.e4m3_quantize(blk)
        assert np.array_equal(tab[A2[mb * 32:(mb + 1) * 32, kb * 32:(kb + 1) * 32]], blk)
        sA2 = sA.copy()
        sA2[mb, kb] = sA2[mb, kb] / 2
        C1, T1 = oracle.gemm(A2, sA2, B, sB, M, N, K)
        assert np.array_equal(C0, C1)
        assert np.array_equal(T0, T1)
    B2 = B.copy()
    blk = tab[B2[32:64, 0:32]] * 2.0
    B2[32:64, 0:32] = oracle.e4m3_quantize(blk)
    sB2 = sB.copy()
    sB2[1, 0] /= 2
    C2, _ = oracle.gemm(A, sA, B2, sB2, M, N, K)
    assert np.array_equal(C0, C2)


def test_operand_swap_symmetry():
    M, N, K = 45, 70, 96
    A, sA, B, sB = _rand_problem(M, N, K, seed=9, arbitrary=True)
    C, T = oracle.gemm(A, sA, B, sB, M, N, K)
    Ct, Tt = oracle.gemm(B, sB, A, sA, N, M, K)
    assert np.array_equal(C, Ct.T)
    assert np.array_equal(T, Tt.T)


def test_sampled_equals_full_and_threads_do_not_matter():
    M, N, K = 77, 96, 128
    A, sA, B, sB = _rand_problem(M, N, K, seed=10, arbitrary=True)
    C1, T1 = oracle.gemm(A, sA, B, sB, M, N, K, nthreads=1)
    C4, T4 = oracle.gemm(A, sA, B, sB, M, N, K, nthreads=5)
    assert np.array_equal(C1, C4) and np.array_equal(T1, T4)
    rng = np.random.default_rng(10)
    ms = rng.integers(0, M, 300)
    ns = rng.integers(0, N, 300)
    Cs, Ts = oracle.gemm_sampled(A, sA, B, sB, M, N, K, ms, ns)
    assert np.array_equal(Cs, C1[ms, ns]) and np.array_equal(Ts, T1[ms, ns])


def test_zero_sized_and_bad_arguments():
    C, T = oracle.gemm(np.zeros((0, 64), np.uint8), np.zeros((0, 2), np.float32),
                       np.zeros((32, 64), np.uint8), np.ones((1, 2), np.float32), 0, 32, 64)
    assert C.shape == (0, 32)
    with pytest.raises(ValueError):
        oracle.gemm(np.zeros((4, 40), np.uint8), np.ones((1, 1), np.float32),
                    np.zeros((32, 40), np.uint8), np.ones((1, 1), np.float32), 4, 32, 40)


@pytest.mark.parametrize("mutation", [1, 2, 3])
def test_planted_mistakes_are_caught(mutation):
    """Each planted mistake (wrong scale index, dropped K block, missing B
    scale) is caught by the brute-force pin."""
    M, N, K = 40, 66, 96
    A, sA, B, sB = _rand_problem(M, N, K, seed=11, elo=-2, ehi=2)
    C, _ = oracle.gemm(A, sA, B, sB, M, N, K, mutation=mutation)
    Ce, _ = _exact(A, sA, B, sB, M, N, K)
    mismatches = sum(Fraction(C[m, n]) != Ce[m][n] for m in range(M) for n in range(N))
    assert mismatches > 0


# ------------------------------------------------------------- workloads ----

@pytest.mark.parametrize("name", ["c0"])
def test_workload_codes_are_finite_and_cast_like_the_oracle(name):
    p = workloads.make(name, seed=0)
    tab = oracle.e4m3_table()
    for codes in (p.A, p.B):
        c = codes.numpy()
        assert not np.isnan(tab[c]).any()
    s = torch.randn(2000, generator=torch.Generator().manual_seed(0)).clamp(-448, 448)
    ours = oracle.e4m3_quantize(s.double().numpy())
    assert np.array_equal(ours, workloads.to_e4m3_codes(s).numpy())
    # power-of-two scales within the stated exponent range
    for sc in (p.sA, p.sB):
        e = np.log2(sc.numpy())
        assert np.all(e == np.round(e)) and e.min() >= -4 and e.max() <= 4


def test_outlier_workload_quantisation():
    p = workloads.outlier(n=256, seed=0)
    tab = oracle.e4m3_table()
    a = tab[p.A.numpy()]
    assert not np.isnan(a).any()
    # every block reaches the E4M3 maximum (amax/scale = 448) up to rounding
    blocks = np.abs(a).reshape(8, 32, 8, 32).max(axis=(1, 3))
    assert np.all(blocks >= 416) and np.all(blocks <= 448)
    s = p.sA.numpy()
    assert np.mean(s != np.exp2(np.round(np.log2(s)))) > 0.9  # not powers of two


def test_grouped_workload_layout():
    gp = workloads.grouped(seed=0, G=4, N=64, K=128)
    assert gp.A.shape == (sum(gp.Ms), 128)
    assert gp.offsets == [sum(gp.Ms[:g]) for g in range(4)]
    assert all(1 <= m <= 64 for m in gp.Ms)
    for g in range(4):
        assert gp.sA[g].shape == ((gp.Ms[g] + 31) // 32, 4)
        assert gp.B[g].shape == (64, 128) and gp.sB[g].shape == (2, 4)


# ------------------------------------------------------- block quantization

def _bf16_matrix(M, K, seed, outlier_frac=0.005):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, K, generator=g)
    hit = torch.rand(M, K, generator=g) < outlier_frac
    x = torch.where(hit, x * 50.0, x)
    x[:, :32] *= 1e-4                                   # tiny values: subnormal codes
    if M >= 64 and K >= 64:
        x[32:64, 32:64] = 0.0                           # an all-zero block
    return x.to(torch.bfloat16)


def _bits(xb):
    return xb.view(torch.int16).numpy().view(np.uint16)


def test_quantize_matches_library_cast():
    """Pinned to torch's float8_e4m3fn cast (round to nearest-even) of the same
    fp32 quotient, clamped to +-448 first (saturation), with the scale
    amax/448 computed by torch in fp32."""
    M, K = 77, 160
    xb = _bf16_matrix(M, K, seed=11)
    q, s = oracle.quantize_blocks(_bits(xb), M, K)
    xf = xb.float()
    Mp = (M + 31) // 32 * 32
    pad = torch.zeros(Mp, K)
    pad[:M] = xf
    amax = pad.view(Mp // 32, 32, K // 32, 32).abs().amax(dim=(1, 3))
    s_ref = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    full = s_ref.repeat_interleave(32, 0).repeat_interleave(32, 1)[:M]
    q_ref = (xf / full).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(s, s_ref.numpy())
    assert np.array_equal(q, q_ref)


def test_quantize_block_maximum_maps_to_448_and_zero_blocks():
    M, K = 96, 96
    xb = _bf16_matrix(M, K, seed=12)
    q, s = oracle.quantize_blocks(_bits(xb), M, K)
    xf = xb.float().numpy()
    for mb in range(3):
        for kb in range(3):
            blk = xf[32 * mb:32 * mb + 32, 32 * kb:32 * kb + 32]
            qb = q[32 * mb:32 * mb + 32, 32 * kb:32 * kb + 32]
            if not blk.any():
                assert s[mb, kb] == 1.0 and not (qb & 0x7F).any()
                continue
            i = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
            assert qb[i] == (0xFE if blk[i] < 0 else 0x7E)
            assert s[mb, kb] == np.float32(np.abs(blk).max()) / np.float32(448.0)


def test_quantize_power_of_two_rescaling():
    """x * 2^j (exact in bf16) gives the same codes and, for blocks that are
    not all zero (their scale stays 1), scales * 2^j."""
    M, K = 64, 64
    xb = _bf16_matrix(M, K, seed=13, outlier_frac=0.0)
    q0, s0 = oracle.quantize_blocks(_bits(xb), M, K)
    zero = ~xb.float().view(2, 32, 2, 32).abs().amax(dim=(1, 3)).bool().numpy()
    assert zero.any() and not zero.all()
    for j in (-3, 5):
        xj = (xb.float() * 2.0 ** j).to(torch.bfloat16)
        assert torch.equal(xj.float(), xb.float() * 2.0 ** j)
        qj, sj = oracle.quantize_blocks(_bits(xj), M, K)
        assert np.array_equal(qj, q0)
        assert np.array_equal(sj, np.where(zero, np.float32(1.0), s0 * np.float32(2.0 ** j)))


# ------------------------------------------------ per-token x per-channel

def test_rowcol_per_tensor_closed_form():
    """Constant vectors (a per-tensor scale): alpha*beta times numpy's fp64
    matmul of the decoded operands, exact here (partial sums are multiples of
    2^-18 below 2^35)."""
    M, N, K = 45, 64, 320
    A, _, B, _ = _rand_problem(M, N, K, seed=21)
    tab = oracle.e4m3_table()
    alpha, beta = np.float32(0.3), np.float32(1.7)
    C, T = oracle.gemm_rowcol(A, np.full(M, alpha), B, np.full(N, beta), M, N, K)
    prod = tab[A] @ tab[B].T
    assert np.array_equal(C, (float(alpha) * float(beta)) * prod)
    assert np.array_equal(T, (float(alpha) * float(beta)) * (np.abs(tab[A]) @ np.abs(tab[B]).T))


def test_rowcol_identity_and_one_hot():
    """B = identity gives C[m,n] = sA[m]*sB[n]*A[m,n]; a one-hot A row picks
    one column of B."""
    M, K = 40, 64
    N = K
    rng = np.random.default_rng(22)
    A, _, _, _ = _rand_problem(M, N, K, seed=22)
    B = np.zeros((N, K), dtype=np.uint8)
    B[np.arange(N), np.arange(K)] = 0x38                        # 1.0
    sA = (rng.random(M) * 4 - 2).astype(np.float32)              # includes negative scales
    sB = (rng.random(N) * 3).astype(np.float32)
    tab = oracle.e4m3_table()
    C, _ = oracle.gemm_rowcol(A, sA, B, sB, M, N, K)
    assert np.array_equal(C, (sA.astype(np.float64)[:, None] * sB.astype(np.float64)[None, :]) * tab[A])
    A1 = np.zeros((M, K), dtype=np.uint8)
    ks = rng.integers(0, K, M)
    A1[np.arange(M), ks] = 0x40                                  # 2.0
    _, _, B2, _ = _rand_problem(M, 96, K, seed=23)
    sB2 = (rng.random(96) + 0.5).astype(np.float32)
    C1, _ = oracle.gemm_rowcol(A1, sA, B2, sB2, M, 96, K)
    for m in range(M):
        exp = (float(sA[m]) * sB2.astype(np.float64)) * 2.0 * tab[B2[:, ks[m]]]
        assert np.array_equal(C1[m], exp)


def test_rowcol_agrees_with_block_oracle_on_block_constant_scales():
    """Scales constant over 32-row and 32-column blocks are also 32x32 block
    scales: the separately pinned block-scaled oracle must agree within its
    fp64 rounding (one rounding per K block there, none here)."""
    M, N, K = 64, 96, 256
    A, _, B, _ = _rand_problem(M, N, K, seed=24)
    rng = np.random.default_rng(24)
    a = (rng.random(M // 32) * 2 + 0.1).astype(np.float32)
    b = (rng.random(N // 32) * 2 + 0.1).astype(np.float32)
    Cr, Tr = oracle.gemm_rowcol(A, np.repeat(a, 32), B, np.repeat(b, 32), M, N, K)
    Cb, Tb = oracle.gemm(A, np.repeat(a[:, None], K // 32, axis=1), B, np.repeat(b[:, None], K // 32, axis=1), M, N, K)
    assert np.all(np.abs(Cr - Cb) <= 1e-12 * Tr)
    assert np.allclose(Tr, Tb, rtol=1e-12, atol=0)


def test_rowcol_operand_swap_symmetry():
    M, N, K = 33, 64, 96
    A, _, B, _ = _rand_problem(M, N, K, seed=25)
    rng = np.random.default_rng(25)
    sA = rng.random(M).astype(np.float32)
    sB = rng.random(N).astype(np.float32)
    C, _ = oracle.gemm_rowcol(A, sA, B, sB, M, N, K)
    Ct, _ = oracle.gemm_rowcol(B, sB, A, sA, N, M, K)
    assert np.array_equal(C, Ct.T)


# -------------------------------------------------------- GEMM + residual ----

def _bf16_bits_of(x):
    """bf16 bit patterns of fp32 values via torch's cast (not the oracle)."""
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy()


def test_residual_zero_reduces_to_gemm():
    M, N, K = 45, 64, 160
    A, sA, B, sB = _rand_problem(M, N, K, seed=21, arbitrary=True)
    R = np.zeros((M, N), dtype=np.uint16)
    C0, T0 = oracle.gemm(A, sA, B, sB, M, N, K)
    C1, T1 = oracle.gemm_residual(A, sA, B, sB, R, M, N, K)
    assert np.array_equal(C0, C1) and np.array_equal(T0, T1)
    # -0.0 (0x8000) is a zero residual too
    C2, _ = oracle.gemm_residual(A, sA, B, sB, np.full((M, N), 0x8000, np.uint16), M, N, K)
    assert np.array_equal(C0, C2)


def _identity_case(M, K, seed):
    A, _, _, _ = _rand_problem(M, K, K, seed=seed)
    B = np.zeros((K, K), dtype=np.uint8)
    B[np.arange(K), np.arange(K)] = 0x38                          # 1.0
    ones_a = np.ones(((M + 31) // 32, K // 32), np.float32)
    ones_b = np.ones((K // 32, K // 32), np.float32)
    rng = np.random.default_rng(seed)
    R = _bf16_bits_of(rng.standard_normal((M, K)) * 30)
    # closed form from torch's own decodings: C = A + R, one fp64 rounding
    a = torch.from_numpy(A).view(torch.float8_e4m3fn).to(torch.float64)
    r = torch.from_numpy(R).view(torch.bfloat16).to(torch.float64)
    return A, ones_a, B, ones_b, R, (a + r).numpy()


def test_residual_identity_weights_closed_form():
    M, K = 70, 96
    A, sA, B, sB, R, exp = _identity_case(M, K, seed=22)
    C, _ = oracle.gemm_residual(A, sA, B, sB, R, M, K, K)
    assert np.array_equal(C, exp)


@pytest.mark.parametrize("mutation", [4, 5])
def test_residual_planted_mistakes_are_caught(mutation):
    """A dropped residual or one taken from the wrong column fails the
    identity-weights closed form."""
    M, K = 40, 64
    A, sA, B, sB, R, exp = _identity_case(M, K, seed=23)
    C, _ = oracle.gemm_residual(A, sA, B, sB, R, M, K, K, mutation=mutation)
    assert not np.array_equal(C, exp)


def test_residual_sampled_equals_full():
    M, N, K = 77, 96, 128
    A, sA, B, sB = _rand_problem(M, N, K, seed=24, arbitrary=True)
    R = _bf16_bits_of(np.random.default_rng(24).standard_normal((M, N)) * 5)
    C, T = oracle.gemm_residual(A, sA, B, sB, R, M, N, K)
    rng = np.random.default_rng(25)
    ms = rng.integers(0, M, 300)
    ns = rng.integers(0, N, 300)
    Cs, Ts = oracle.gemm_residual_sampled(A, sA, B, sB, R, M, N, K, ms, ns)
    assert np.array_equal(Cs, C[ms, ns]) and np.array_equal(Ts, T[ms, ns])


# ----------------------------------------------------- per-token A scales ----

def test_pertoken_with_block_constant_scales_equals_block_oracle():
    """Per-row scales equal within each 32-row block are the 32x32 block
    case: the two oracles agree exactly."""
    M, N, K = 70, 64, 160
    A, sA, B, sB = _rand_problem(M, N, K, seed=31, arbitrary=True)
    sA_tok = np.repeat(sA, 32, axis=0)[:M]
    C1, T1 = oracle.gemm(A, sA, B, sB, M, N, K)
    C2, T2 = oracle.gemm_pertoken(A, sA_tok, B, sB, M, N, K)
    assert np.array_equal(C1, C2) and np.array_equal(T1, T2)


def test_pertoken_brute_force_exact():
    """Distinct power-of-two scales per row: every partial sum is exact, and
    the oracle equals exact rational arithmetic; a per-row scale read from
    the wrong row (mutation 6) fails it."""
    M, N, K = 37, 33, 96
    rng = np.random.default_rng(32)
    A, _, B, sB = _rand_problem(M, N, K, seed=32, elo=-2, ehi=2)
    sA = np.ldexp(1.0, rng.integers(-2, 3, (M, K // 32))).astype(np.float32)
    tab = oracle.e4m3_table()
    C, _ = oracle.gemm_pertoken(A, sA, B, sB, M, N, K)
    Cm, _ = oracle.gemm_pertoken(A, sA, B, sB, M, N, K, mutation=6)
    mismatches = 0
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(sA[m, k // 32])) * Fraction(float(sB[n // 32, k // 32]))
                        * Fraction(tab[A[m, k]]) * Fraction(tab[B[n, k]]) for k in range(K))
            assert Fraction(C[m, n]) == exact
            mismatches += Fraction(Cm[m, n]) != exact
    assert mismatches > 0


def test_pertoken_row_scaling_closed_form():
    """Scales constant along K for each row (per token) and unit B scales:
    C = diag(sA) (A B^T), the fp64 matmul of the decoded codes (exact)."""
    M, N, K = 45, 64, 128
    A, _, B, _ = _rand_problem(M, N, K, seed=33)
    rng = np.random.default_rng(33)
    a = np.ldexp(1.0, rng.integers(-5, 6, M))
    sA = np.repeat(a[:, None], K // 32, axis=1).astype(np.float32)
    sB = np.ones((N // 32, K // 32), np.float32)
    tab = oracle.e4m3_table()
    C, _ = oracle.gemm_pertoken(A, sA, B, sB, M, N, K)
    assert np.array_equal(C, a[:, None] * (tab[A] @ tab[B].T))
