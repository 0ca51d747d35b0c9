"""Bounded waits: a withheld pipeline stage makes the kernel's waits run out;
the kernel records FP8_ERR_TIMEOUT in the device status word and returns
cleanly, and the context stays usable for a normal call afterwards.  No GPU
fault is involved: every wait in the kernel has an iteration budget."""
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
    return mod


@pytest.mark.parametrize("grouped", [False, True])
def test_withheld_stage_times_out_cleanly(bs, grouped):
    p = workloads.square(n=512, seed=1)
    A, sA, B, sB = p.A.to(DEV), p.sA.to(DEV), p.B.to(DEV), p.sB.to(DEV)
    C = torch.empty(p.M, p.N, dtype=torch.bfloat16, device=DEV)
    assert bs.fp8_status_query() == 0
    bs.fp8_debug_set(bs.FP8_DEBUG_WAIT_LIMIT_CYCLES, 20_000_000)   # ~10 ms
    bs.fp8_debug_set(bs.FP8_DEBUG_WITHHOLD_STAGE, 1)
    try:
        if grouped:
            Ms = torch.tensor([p.M], dtype=torch.int32, device=DEV)
            bs.fp8_gemm_grouped([(A, sA, B, sB, C)], Ms, p.N, p.K)
        else:
            bs.fp8_gemm_blockscaled(A, sA, B, sB, C, p.M, p.N, p.K)
        torch.cuda.synchronize()
        assert bs.fp8_status_query() == bs._abi.FP8_ERR_TIMEOUT
    finally:
        bs.fp8_debug_set(bs.FP8_DEBUG_WITHHOLD_STAGE, -1)
        bs.fp8_debug_set(bs.FP8_DEBUG_WAIT_LIMIT_CYCLES, 0)
    # the context is intact and the next call is correct
    bs.fp8_gemm_blockscaled(A, sA, B, sB, C, p.M, p.N, p.K)
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == 0
    Cr, T = oracle.gemm(p.A.numpy(), p.sA.numpy(), p.B.numpy(), p.sB.numpy(), p.M, p.N, p.K)
    check(bf16_to_f64(C), Cr, T, "after timeout")
