"""Grouped decode under CUDA-graph replay.

The group row counts live in device memory and are read only by the kernel,
so one captured launch serves any later counts: between replays the test
rewrites the counts in place and checks every group against the oracle, and
that nothing is written past a group's current row count (FP8 GEMM library
article, hncyxsy.com/news/241433, section 4.3: shapes in device memory so a
captured graph stays valid)."""
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


def test_graph_replay_follows_device_row_counts(bs):
    G, N, K, CAP = 5, 288, 480, 64
    gp = workloads.grouped(seed=7, G=G, N=N, K=K, Ms=[CAP] * G)   # CAP rows of capacity per group
    A = [gp.A_group(g).to(DEV) for g in range(G)]
    sA = [s.to(DEV) for s in gp.sA]
    B = [b.to(DEV) for b in gp.B]
    sB = [s.to(DEV) for s in gp.sB]
    C = [torch.full((CAP + 1, N), -7.0, dtype=torch.bfloat16, device=DEV) for _ in range(G)]
    Ms = torch.full((G,), CAP, dtype=torch.int32, device=DEV)
    groups = [(A[g], sA[g], B[g], sB[g], C[g]) for g in range(G)]

    bs.fp8_gemm_grouped(groups, Ms, N, K)   # device set-up happens outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        bs.fp8_gemm_grouped(groups, Ms, N, K)

    for counts in ([CAP] * G, [1, 33, 0, 64, 7], [17, 2, 64, 1, 40]):
        for c in C:
            c.fill_(-7.0)
        Ms.copy_(torch.tensor(counts, dtype=torch.int32))
        graph.replay()
        torch.cuda.synchronize()
        for g, m in enumerate(counts):
            assert torch.all(C[g][m:] == -7.0), f"counts {counts}: group {g} written past row {m}"
            if m == 0:
                continue
            Cr, T = oracle.gemm(gp.A_group(g)[:m].numpy(), gp.sA[g][:(m + 31) // 32].numpy(),
                                gp.B[g].numpy(), gp.sB[g].numpy(), m, N, K)
            check(bf16_to_f64(C[g][:m]), Cr, T, f"graph replay {counts} g{g}")
    assert bs.fp8_status_query() == 0
