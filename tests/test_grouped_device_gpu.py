"""Grouped GEMM with device-resident group records (fp8_gemm_grouped_device,
through the C ABI): the records, row counts and tensor maps all live in
device memory, so a CUDA graph captured once computes whatever problems the
table holds at each replay (FP8 GEMM library article, hncyxsy.com/news/241433,
section 4.2 "parameter table", section 4.3 "CUDA Graph").  Checked against
the host-table call bit for bit and against the oracle."""
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


def _device_problem(gp, sentinel=-7.0):
    """The group tensors on the device and each group's output with one
    sentinel row past M_g."""
    A = gp.A.to(DEV)
    groups, outs = [], []
    for g in range(gp.G):
        o, m = gp.offsets[g], gp.Ms[g]
        C = torch.full((max(m, 1) + 1, gp.N), sentinel, dtype=torch.bfloat16, device=DEV)
        outs.append(C)
        groups.append((A[o:o + m] if m else A, gp.sA[g].to(DEV) if gp.sA[g].numel() else gp.sB[g].to(DEV),
                       gp.B[g].to(DEV), gp.sB[g].to(DEV), C))
    return groups, outs


def _oracle_check(gp, outs, what):
    for g in range(gp.G):
        if gp.Ms[g] == 0:
            continue
        Cr, T = oracle.gemm(gp.A_group(g).numpy(), gp.sA[g].numpy(), gp.B[g].numpy(), gp.sB[g].numpy(),
                            gp.Ms[g], gp.N, gp.K)
        check(bf16_to_f64(outs[g][:gp.Ms[g]]), Cr, T, f"{what} group {g}")


def test_device_table_equals_host_table(bs):
    gp = workloads.grouped(seed=21, G=6, N=288, K=416, Ms=[0, 1, 33, 130, 64, 200])
    groups, outs = _device_problem(gp)
    Ms = torch.tensor(gp.Ms, dtype=torch.int32, device=DEV)
    table = bs.group_table(groups, DEV)
    ws = torch.empty(bs.fp8_grouped_workspace_bytes(gp.G), dtype=torch.uint8, device=DEV)
    bs.fp8_gemm_grouped_device(table, Ms, gp.N, gp.K, ws)
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == 0
    ref = [torch.empty_like(o) for o in outs]
    bs.fp8_gemm_grouped([(a, sa, b, sb, c) for (a, sa, b, sb, _), c in zip(groups, ref)], Ms, gp.N, gp.K)
    torch.cuda.synchronize()
    for g in range(gp.G):
        m = gp.Ms[g]
        assert torch.all(outs[g][m:] == -7.0), f"group {g}: store past M_g"
        assert torch.equal(outs[g][:m].view(torch.int16), ref[g][:m].view(torch.int16)), f"group {g}"
    _oracle_check(gp, outs, "device table")


def test_graph_replay_follows_new_pointers_and_row_counts(bs):
    """One capture; between replays the table is rewritten with other
    buffers (other A, B, C pointers) and other row counts."""
    N, K, G = 256, 320, 4
    gp1 = workloads.grouped(seed=22, G=G, N=N, K=K, Ms=[5, 64, 17, 1])
    gp2 = workloads.grouped(seed=23, G=G, N=N, K=K, Ms=[40, 0, 3, 64])
    g1, o1 = _device_problem(gp1)
    g2, o2 = _device_problem(gp2)
    t1, t2 = bs.group_table(g1, DEV), bs.group_table(g2, DEV)
    m1 = torch.tensor(gp1.Ms, dtype=torch.int32, device=DEV)
    m2 = torch.tensor(gp2.Ms, dtype=torch.int32, device=DEV)
    table = t1.clone()
    Ms = m1.clone()
    ws = torch.empty(bs.fp8_grouped_workspace_bytes(G), dtype=torch.uint8, device=DEV)
    bs.fp8_gemm_grouped_device(table, Ms, N, K, ws)   # set-up outside the capture
    torch.cuda.synchronize()
    for o in o1:
        o.fill_(-7.0)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        bs.fp8_gemm_grouped_device(table, Ms, N, K, ws)
    graph.replay()
    torch.cuda.synchronize()
    _oracle_check(gp1, o1, "replay 1")
    first = [o.clone() for o in o1]
    table.copy_(t2)
    Ms.copy_(m2)
    graph.replay()
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == 0
    _oracle_check(gp2, o2, "replay 2")
    for g in range(G):
        assert torch.all(o2[g][gp2.Ms[g]:] == -7.0), f"group {g}: store past M_g"
        assert torch.equal(o1[g].view(torch.int16), first[g].view(torch.int16)), "replay 2 wrote old buffers"
    del graph


def test_rejected_record_is_skipped_and_reported(bs):
    gp = workloads.grouped(seed=24, G=3, N=128, K=256, Ms=[20, 33, 9])
    groups, outs = _device_problem(gp)
    table = bs.group_table(groups, DEV)
    table[1, 0] += 1   # group 1's A is no longer 16-byte aligned
    Ms = torch.tensor(gp.Ms, dtype=torch.int32, device=DEV)
    ws = torch.empty(bs.fp8_grouped_workspace_bytes(gp.G), dtype=torch.uint8, device=DEV)
    bs.fp8_gemm_grouped_device(table, Ms, gp.N, gp.K, ws)
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == bs._abi.FP8_ERR_RECORD
    assert bs.fp8_status_query() == 0
    assert torch.all(outs[1] == -7.0), "a rejected group was written"
    for g in (0, 2):
        Cr, T = oracle.gemm(gp.A_group(g).numpy(), gp.sA[g].numpy(), gp.B[g].numpy(), gp.sB[g].numpy(),
                            gp.Ms[g], gp.N, gp.K)
        check(bf16_to_f64(outs[g][:gp.Ms[g]]), Cr, T, f"rejected-record launch group {g}")


def test_more_groups_than_one_launch(bs):
    G = 70
    rng = np.random.default_rng(25)
    Ms_list = [int(m) for m in rng.integers(0, 40, G)]
    gp = workloads.grouped(seed=25, G=G, N=64, K=96, Ms=Ms_list)
    groups, outs = _device_problem(gp)
    Ms = torch.tensor(gp.Ms, dtype=torch.int32, device=DEV)
    table = bs.group_table(groups, DEV)
    ws = torch.empty(bs.fp8_grouped_workspace_bytes(G), dtype=torch.uint8, device=DEV)
    bs.fp8_gemm_grouped_device(table, Ms, gp.N, gp.K, ws)
    torch.cuda.synchronize()
    assert bs.fp8_status_query() == 0
    ref = [torch.empty_like(o) for o in outs]
    bs.fp8_gemm_grouped([(a, sa, b, sb, c) for (a, sa, b, sb, _), c in zip(groups, ref)], Ms, gp.N, gp.K)
    torch.cuda.synchronize()
    for g in range(G):
        m = gp.Ms[g]
        assert torch.equal(outs[g][:m].view(torch.int16), ref[g][:m].view(torch.int16)), f"group {g}"
