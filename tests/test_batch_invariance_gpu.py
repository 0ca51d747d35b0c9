"""Batch invariance when the scale kinds mix inside one output tile.

A row's result may not depend on how many other rows share its launch ("AI
Infra 进阶：如何让大模型输出确定的结果", aif.amtbbs.org post 29992, section 1:
only a batch-dependent reduction split changes a row's bits).  The K order
of every path is fixed, so only the choice of path can depend on the other
rows: under FP8_PATH_AUTO a tile takes the block-scaled MMA when every scale
it reads is a power of two, and the rows of one tile share that choice.

The contract checked here (and stated in include/bsfp8.h):
  * FP8_PATH_PROMOTE gives each row the same bits for every M, whatever the
    scales;
  * FP8_PATH_AUTO does the same whenever sA's 32-row blocks are all of one
    kind (every block's scales all powers of two, or every block holding at
    least one that is not); sB may mix freely, since every launch reads the
    same sB;
  * when sA's row blocks mix kinds inside one tile, AUTO's bits for a row may
    change with M, but they are always those of one of the two pinned paths,
    and within the tolerance of the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._accept import bf16_to_f64, check

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SIZES = (1, 7, 64, 8192)
M_FULL, N, K = 8192, 512, 1024


@pytest.fixture(scope="module")
def bs():
    import block_scaled_fp8_sm_gb300 as mod
    from block_scaled_fp8_sm_gb300 import build
    build.build()
    mod.library()
    return mod


def _base(seed):
    g = torch.Generator().manual_seed(seed)
    A = workloads.normal_codes(M_FULL, K, g, "cpu")
    B = workloads.normal_codes(N, K, g, "cpu")
    sA = workloads.pow2_scales(M_FULL, K // 32, -3, 3, g, "cpu")
    sB = workloads.pow2_scales(N, K // 32, -3, 3, g, "cpu")
    return A, sA, B, sB


def _mixed_a(seed):
    """Row blocks 0 and 1 (rows 0-63) keep power-of-two scales; row block 3
    (rows 96-127, the same 256-row tile) and one block in every later tile get
    one scale multiplied by 1.3."""
    A, sA, B, sB = _base(seed)
    sA[3, 5] *= 1.3
    for rb in range(8 + 2, sA.shape[0], 8):
        sA[rb, (rb * 7) % (K // 32)] *= 1.3
    return A, sA, B, sB


def _mixed_b(seed):
    """sA all powers of two; sB has non-power-of-two scales in the first
    256-column tile only (that tile promotes, the second one does not)."""
    A, sA, B, sB = _base(seed)
    sB[1, 3] *= 1.3
    sB[6, 30] *= 0.7
    return A, sA, B, sB


def _rows(bs, A, sA, B, sB, m, mode):
    dA = A[:m].contiguous().to(DEV)
    dsA = sA[:(m + 31) // 32].contiguous().to(DEV)
    C = torch.empty(m, N, dtype=torch.bfloat16, device=DEV)
    bs.fp8_gemm_blockscaled(dA, dsA, B.to(DEV), sB.to(DEV), C, m, N, K, mode=mode)
    torch.cuda.synchronize()
    return C[:64].view(torch.int16).cpu().clone()


def _oracle_check(A, sA, B, sB, bits, what):
    Cr, T = oracle.gemm(A[:64].numpy(), sA[:2].numpy(), B.numpy(), sB.numpy(), 64, N, K)
    check(bf16_to_f64(bits.view(torch.bfloat16)), Cr, T, what)


def test_promote_is_batch_invariant_with_mixed_row_blocks(bs):
    A, sA, B, sB = _mixed_a(41)
    rows = {m: _rows(bs, A, sA, B, sB, m, bs.FP8_PATH_PROMOTE) for m in SIZES}
    ref = rows[M_FULL]
    for m in SIZES:
        k = min(m, 64)
        assert torch.equal(rows[m][:k], ref[:k]), f"PROMOTE: M={m} differs from M={M_FULL}"
    _oracle_check(A, sA, B, sB, ref, "mixed sA, PROMOTE")
    assert bs.fp8_status_query() == 0


def test_auto_is_batch_invariant_when_sa_row_blocks_share_a_kind(bs):
    A, sA, B, sB = _mixed_b(42)
    rows = {m: _rows(bs, A, sA, B, sB, m, None) for m in SIZES}
    ref = rows[M_FULL]
    for m in SIZES:
        k = min(m, 64)
        assert torch.equal(rows[m][:k], ref[:k]), f"AUTO (mixed sB only): M={m} differs"
    _oracle_check(A, sA, B, sB, ref, "mixed sB, AUTO")
    assert bs.fp8_status_query() == 0


def test_auto_with_mixed_row_blocks_takes_one_of_the_pinned_paths(bs):
    """Rows 0-63 sit in a 256-row tile whose row block 3 is not all powers of
    two: a launch of M >= 97 promotes that tile, a launch of M <= 64 does not
    see block 3 and runs the block-scaled MMA."""
    A, sA, B, sB = _mixed_a(43)
    promoted = _rows(bs, A, sA, B, sB, M_FULL, bs.FP8_PATH_PROMOTE)
    for m in SIZES:
        auto = _rows(bs, A, sA, B, sB, m, None)
        k = min(m, 64)
        if m > 96:
            assert torch.equal(auto[:k], promoted[:k]), f"M={m}: AUTO differs from PROMOTE"
        else:
            native = _rows(bs, A, sA, B, sB, m, bs.FP8_PATH_NATIVE)
            assert torch.equal(auto[:k], native[:k]), f"M={m}: AUTO differs from NATIVE"
        if m == 64 or m == M_FULL:
            _oracle_check(A, sA, B, sB, auto, f"mixed sA, AUTO, M={m}")
    assert bs.fp8_status_query() == 0
