"""Benchmark of the block-scaled E4M3 GEMM library on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one block-scaled GEMM of the headline workload, the prefill
projection M=8192, N=28672, K=8192 (power-of-two 32x32 scales, bf16 out), with
inputs resident in HBM; the L2 is flushed (a 512 MiB write) between timed
steps and each step is timed with CUDA events on the launching stream.  The
same JSON line also carries the other workloads measured the same way: the
M=N=K=4096 square GEMM, the grouped decode batch (G=16, M_g in [1,64], N=4096,
K=7168; GB/s against HBM; also as a CUDA-graph replay; its 470 MB of weights
per step exceed the L2, so it runs without the flush, and its read-flushed and
write-flushed times are reported beside it), the 8192^3 arbitrary-scale GEMM
with outliers (promotion path; also with the path pinned), the block
quantization of 8192x8192 bf16 activations (GB/s against HBM), the 4096^3 GEMM
with per-token x per-channel scales, the 4096^3 GEMM with a fused residual
add, the per-token-scale 4096^3 GEMMs (fp32 scales, and UE8M0 bytes), and the
prefill GEMM with its output quantized to E4M3 in the epilogue (beside the same
work unfused: the bf16 GEMM followed by the block quantizer).  Every generated input buffer is recorded by
its SHA-256, with the torch version that generated it.

``--impl reference`` times the CPU oracle (the only other implementation of
the method; plain C, fp64) on a bounded sample of the same workload.

Multi-GPU: the GEMM runs as independent replicas, one per rank (weak scaling);
ranks only meet for the timing barrier and the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

MEASURED = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_PER_BF16 = 2.0   # nominal dense ratio (4.5 / 2.25 PFLOP/s)
L2_FLUSH_BYTES = 512 << 20

HEADLINE = "c2"
HEADLINE_SHAPE = {"M": 8192, "N": 28672, "K": 8192}
WORKLOAD_NAMES = {
    "c1": "block-scaled E4M3 GEMM M=N=K=4096, pow2 32x32 scales, bf16 out",
    "c2": "prefill projection GEMM M=8192 N=28672 K=8192, pow2 32x32 scales",
    "c3": "grouped decode G=16 M_g~U[1,64] N=4096 K=7168, per-group B, pow2 scales",
    "c4": "arbitrary-scale GEMM M=N=K=8192 (amax/448 scales, 0.5% x50 outliers)",
    "c4p": "arbitrary-scale GEMM M=N=K=8192 as c4, promotion path pinned (mode PROMOTE: single-CTA tiles)",
    "q8": "block quantization of bf16 activations 8192x8192 -> E4M3 codes + 32x32 fp32 scales",
    "r1": "per-token x per-channel scaled E4M3 GEMM M=N=K=4096 (fp32 scales [M] and [N]), bf16 out",
    "f1": "block-scaled E4M3 GEMM M=N=K=4096 with a bf16 residual added in the epilogue",
    "p1e": ("per-token A scales as UE8M0 bytes (one per row per 32-K block) x 32x32 pow2 B blocks, "
            "E4M3 GEMM M=N=K=4096 (native path), bf16 out"),
    "qo": ("block-scaled E4M3 GEMM M=8192, N=28672, K=8192 (pow2 32x32 scales) whose output is quantized "
           "in the epilogue to E4M3 codes + 32x32 fp32 scales"),
    "p1": "per-token A scales (one fp32 per row per 32-K block) x 32x32 B blocks, E4M3 GEMM M=N=K=4096, bf16 out",
    "p1n": "per-token power-of-two A scales (one per row per 32-K block, UE8M0 on the MMA) x 32x32 pow2 B blocks, "
           "E4M3 GEMM M=N=K=4096 (mode NATIVE), bf16 out",
}


def peaks():
    src = "measured"
    try:
        with open(MEASURED) as f:
            p = json.load(f)
    except Exception:
        p, src = dict(FALLBACK), "fallback"
    return p, src


def _code_only(src):
    """The source without comments and blank lines (no string literal in the
    CUDA sources holds a comment marker), so that editing a comment does not
    count as a kernel change."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.split("\n") if line.strip())


def source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_scaled_fp8_sm_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the kernel source as it is now."""
    try:
        with open(TRAFFIC) as f:
            t = json.load(f)
    except Exception:
        return None
    e = t.get(workload)
    if not e or e.get("source_hash") != source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_init():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- ours ----

def sha256_of(t):
    """SHA-256 of a tensor's bytes (a list of tensors: of their bytes in order)."""
    import torch
    h = hashlib.sha256()
    for x in (t if isinstance(t, (list, tuple)) else [t]):
        h.update(x.detach().contiguous().view(-1).view(torch.uint8).cpu().numpy().tobytes())
    return h.hexdigest()


def make_runner(name, dev, bs):
    """Returns (run(stream), flops, algorithmic bytes, input buffers) for one
    workload with its inputs on the device."""
    import torch

    import workloads
    if name == "q8":
        M = K = 8192
        g = torch.Generator(device=dev).manual_seed(0)
        x = torch.randn(M, K, generator=g, device=dev)
        x = torch.where(torch.rand(M, K, generator=g, device=dev) < 0.005, x * 50.0, x).to(torch.bfloat16)
        q = torch.empty(M, K, dtype=torch.uint8, device=dev)
        sc = torch.empty(M // 32, K // 32, dtype=torch.float32, device=dev)
        nbytes = 2 * M * K + M * K + 4 * sc.numel()

        def run(stream):
            bs.fp8_quantize_blocks(x, q, sc, stream=stream)
        return run, 0, nbytes, {"x": x}
    if name in ("qo", "qo_chain"):
        # the prefill GEMM with its output quantized for the next layer: fused in the
        # epilogue (qo), or the bf16 GEMM followed by the block quantizer (qo_chain)
        p = workloads.make("c2", seed=0, device=dev)
        Cq = torch.empty(p.M, p.N, dtype=torch.uint8, device=dev)
        sC = torch.empty(p.M // 32, p.N // 32, dtype=torch.float32, device=dev)
        nbytes = p.M * p.K + p.N * p.K + 4 * (p.sA.numel() + p.sB.numel()) + p.M * p.N + 4 * sC.numel()
        if name == "qo":
            def run(stream):
                bs.fp8_gemm_blockscaled_quant(p.A, p.sA, p.B, p.sB, Cq, sC, p.M, p.N, p.K, stream=stream)
        else:
            C = torch.empty(p.M, p.N, dtype=torch.bfloat16, device=dev)

            def run(stream):
                bs.fp8_gemm_blockscaled(p.A, p.sA, p.B, p.sB, C, p.M, p.N, p.K, stream=stream)
                bs.fp8_quantize_blocks(C, Cq, sC, stream=stream)
        return run, p.flops, nbytes, {"A": p.A, "sA": p.sA, "B": p.B, "sB": p.sB}
    if name == "f1":
        p = workloads.make("c1", seed=0, device=dev)
        g = torch.Generator(device=dev).manual_seed(1)
        R = torch.randn(p.M, p.N, generator=g, device=dev).to(torch.bfloat16)
        C = torch.empty(p.M, p.N, dtype=torch.bfloat16, device=dev)

        def run(stream):
            bs.fp8_gemm_blockscaled_residual(p.A, p.sA, p.B, p.sB, R, C, p.M, p.N, p.K, stream=stream)
        return run, p.flops, p.algorithmic_bytes + 2 * p.M * p.N, {"A": p.A, "sA": p.sA, "B": p.B, "sB": p.sB, "R": R}
    if name == "p1e":
        p = workloads.make("c1", seed=0, device=dev)
        g = torch.Generator(device=dev).manual_seed(2)
        e = torch.randint(127 - 4, 127 + 5, (p.M, p.K // 32), generator=g, device=dev).to(torch.uint8)
        C = torch.empty(p.M, p.N, dtype=torch.bfloat16, device=dev)
        nbytes = p.M * p.K + p.N * p.K + e.numel() + 4 * p.sB.numel() + 2 * p.M * p.N

        def run(stream):
            bs.fp8_gemm_pertoken_e8m0(p.A, e, p.B, p.sB, C, p.M, p.N, p.K, stream=stream)
        return run, p.flops, nbytes, {"A": p.A, "sA": e, "B": p.B, "sB": p.sB}
    if name in ("p1", "p1n"):
        p = workloads.make("c1", seed=0, device=dev)
        g = torch.Generator(device=dev).manual_seed(2)
        if name == "p1":
            sA = torch.rand(p.M, p.K // 32, generator=g, device=dev) + 0.05
            sB = torch.rand(p.N // 32, p.K // 32, generator=g, device=dev) + 0.05
            mode = None
        else:
            sA = torch.ldexp(torch.ones(p.M, p.K // 32, device=dev),
                             torch.randint(-4, 5, (p.M, p.K // 32), generator=g, device=dev)).float()
            sB = p.sB
            mode = bs.FP8_PATH_NATIVE
        C = torch.empty(p.M, p.N, dtype=torch.bfloat16, device=dev)
        nbytes = p.M * p.K + p.N * p.K + 4 * (sA.numel() + sB.numel()) + 2 * p.M * p.N

        def run(stream):
            bs.fp8_gemm_pertoken(p.A, sA, p.B, sB, C, p.M, p.N, p.K, stream=stream, mode=mode)
        return run, p.flops, nbytes, {"A": p.A, "sA": sA, "B": p.B, "sB": sB}
    if name == "r1":
        p = workloads.make("c1", seed=0, device=dev)
        g = torch.Generator(device=dev).manual_seed(1)
        sA = torch.rand(p.M, generator=g, device=dev) + 0.5
        sB = torch.rand(p.N, generator=g, device=dev) + 0.5
        C = torch.empty(p.M, p.N, dtype=torch.bfloat16, device=dev)
        nbytes = p.M * p.K + p.N * p.K + 4 * (p.M + p.N) + 2 * p.M * p.N

        def run(stream):
            bs.fp8_gemm_rowcol(p.A, sA, p.B, sB, C, p.M, p.N, p.K, stream=stream)
        return run, p.flops, nbytes, {"A": p.A, "sA": sA, "B": p.B, "sB": sB}
    p = workloads.make("c4" if name == "c4p" else name, seed=0, device=dev)
    if name == "c3":
        Cs = [torch.empty(m, p.N, dtype=torch.bfloat16, device=dev) for m in p.Ms]
        groups = [(p.A[o:o + m], sa, b, sb, c) for o, m, sa, b, sb, c in
                  zip(p.offsets, p.Ms, p.sA, p.B, p.sB, Cs)]
        Ms = torch.tensor(p.Ms, dtype=torch.int32, device=dev)

        def run(stream):
            bs.fp8_gemm_grouped(groups, Ms, p.N, p.K, stream=stream)
        return run, p.flops, p.algorithmic_bytes, {"A": p.A, "sA": p.sA, "B": p.B, "sB": p.sB, "Ms": Ms}
    C = torch.empty(p.M, p.N, dtype=torch.bfloat16, device=dev)
    mode = 2 if name == "c4p" else None   # FP8_PATH_PROMOTE

    def run(stream):
        bs.fp8_gemm_blockscaled(p.A, p.sA, p.B, p.sB, C, p.M, p.N, p.K, stream=stream, mode=mode)
    return run, p.flops, p.algorithmic_bytes, {"A": p.A, "sA": p.sA, "B": p.B, "sB": p.sB}


# The HBM-bound workloads move more bytes per step than the 129 MB L2 holds
# (the grouped decode streams 470 MB of weights; the quantizer reads 128 MiB
# and writes 64 MiB), so they run back to back without the write flush: the
# flush leaves L2 full of dirty lines whose write-back then lands inside an
# HBM-bound kernel (~129 MB of extra DRAM writes per step), while a GEMM of the
# square or prefill size is not affected.  Back to back, each step writes back
# only its predecessor's dirty lines, as in a steady stream of steps.  Their
# read-flushed times (a 512 MiB read leaves L2 holding clean lines) and
# write-flushed times are reported beside them.
UNFLUSHED = {"c3": "not flushed: the step's 470 MB of weights exceed the 129 MB L2",
             "q8": "not flushed: the step reads 128 MiB and writes 64 MiB, more than the 129 MB L2"}
# other L2 treatments timed beside the main one, for context
EXTRA_FLUSH = {"c3": ("read", "write"), "q8": ("read", "write")}


def time_device(run, steps, warmup, dev, flush_buf, world, flush="write"):
    """Per-step kernel time (ms) with CUDA events on the launching stream.
    flush: "write" (a 512 MiB fill), "read" (a 512 MiB reduction) or None."""
    import torch
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        run(stream)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    sink = torch.empty((), dtype=torch.int64, device=dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    for i in range(steps):
        if flush == "write":
            flush_buf.fill_(i & 0xFF)      # evict the operands from L2
        elif flush == "read":
            torch.sum(flush_buf.view(torch.int64), dim=(0,), out=sink)
        ev[i][0].record(stream)
        run(stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    return [a.elapsed_time(b) for a, b in ev]


def time_graph_grouped(steps, warmup, dev, bs, flush_buf):
    """The grouped-decode launch captured once in a CUDA graph: device time per
    replay (timed like the direct launch: no L2 flush, the weights exceed L2)
    and host time per launch, direct call versus replay (the direct call
    encodes one tensor map per group)."""
    import torch

    import workloads
    p = workloads.make("c3", seed=0, device=dev)
    Cs = [torch.empty(m, p.N, dtype=torch.bfloat16, device=dev) for m in p.Ms]
    groups = [(p.A[o:o + m], sa, b, sb, c) for o, m, sa, b, sb, c in
              zip(p.offsets, p.Ms, p.sA, p.B, p.sB, Cs)]
    Ms = torch.tensor(p.Ms, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    bs.fp8_gemm_grouped(groups, Ms, p.N, p.K)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        bs.fp8_gemm_grouped(groups, Ms, p.N, p.K)
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in ev) / steps

    def host_us(fn, n=20):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        t1 = time.perf_counter()
        torch.cuda.synchronize(dev)
        return (t1 - t0) / n * 1e6
    direct = host_us(lambda: bs.fp8_gemm_grouped(groups, Ms, p.N, p.K))
    descs = bs.group_descs(groups)
    prebuilt = host_us(lambda: bs.fp8_gemm_grouped(descs, Ms, p.N, p.K))
    replay = host_us(graph.replay)
    del graph

    # the same batch with its records in device memory, captured once: a
    # replay rebuilds the tensor maps from the table on the device first
    table = bs.group_table(groups, dev)
    ws = torch.empty(bs.fp8_grouped_workspace_bytes(len(groups)), dtype=torch.uint8, device=dev)
    bs.fp8_gemm_grouped_device(table, Ms, p.N, p.K, ws)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        bs.fp8_gemm_grouped_device(table, Ms, p.N, p.K, ws)
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize(dev)
    for i in range(steps):
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    ms_dev = sum(a.elapsed_time(b) for a, b in ev) / steps
    replay_dev = host_us(graph.replay)
    del graph
    return {"ms_per_step": round(ms, 4), "value": round(p.algorithmic_bytes / (ms * 1e-3) / 1e9, 1),
            "unit": "GB/s", "host_us_per_launch": {"direct": round(direct, 1), "prebuilt_descs": round(prebuilt, 1),
                                   "graph_replay": round(replay, 1)},
            "device_table_graph_replay": {
                "ms_per_step": round(ms_dev, 4), "value": round(p.algorithmic_bytes / (ms_dev * 1e-3) / 1e9, 1),
                "unit": "GB/s", "host_us_per_replay": round(replay_dev, 1),
                "how": "records, row counts and tensor maps in device memory (fp8_gemm_grouped_device), "
                       "two kernels per replay: tensor-map preparation and the grouped GEMM"}}


def time_e2e(name, steps, warmup, dev, bs, world):
    """Same metric through the public API with pinned HOST buffers, as a
    serving loop runs it: every step copies all of its inputs host->device,
    runs the GEMM and copies all of C back.  Steps are pipelined over three
    streams with double-buffered device memory: step i's C travels back while
    step i+1's inputs come in and its GEMM runs; each step's bytes still move
    inside the timed region."""
    import torch

    import workloads
    p = workloads.make(name, seed=0, device="cpu")
    hA, hsA, hB, hsB = (t.pin_memory() for t in (p.A, p.sA, p.B, p.sB))
    hC = [torch.empty(p.M, p.N, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dev_in = [[torch.empty_like(t, device=dev) for t in (hA, hsA, hB, hsB)] for _ in range(2)]
    dC = [torch.empty(p.M, p.N, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    s_in, s_mm, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "mm", "out")}
    used = [False, False]

    def step(i):
        b = i & 1
        if used[b]:
            s_in.wait_event(ev["mm"][b])        # the GEMM two steps back has read these inputs
        with torch.cuda.stream(s_in):
            for d, h in zip(dev_in[b], (hA, hsA, hB, hsB)):
                d.copy_(h, non_blocking=True)
        ev["in"][b].record(s_in)
        s_mm.wait_event(ev["in"][b])
        if used[b]:
            s_mm.wait_event(ev["out"][b])       # C two steps back has been copied out
        dA, dsA, dB, dsB = dev_in[b]
        bs.fp8_gemm_blockscaled(dA, dsA, dB, dsB, dC[b], p.M, p.N, p.K, stream=s_mm)
        ev["mm"][b].record(s_mm)
        s_out.wait_event(ev["mm"][b])
        with torch.cuda.stream(s_out):
            hC[b].copy_(dC[b], non_blocking=True)
        ev["out"][b].record(s_out)
        used[b] = True

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for i in range(steps):
        step(warmup + i)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_mm)
    t1.record(s_out)
    torch.cuda.synchronize(dev)
    barrier(world)
    ms = t0.elapsed_time(t1) / steps
    h2d = sum(t.numel() * t.element_size() for t in (hA, hsA, hB, hsB))
    d2h = hC[0].numel() * hC[0].element_size()
    return ms, p.flops, h2d, d2h


def time_e2e_grouped(steps, warmup, dev, bs, world):
    """Grouped decode end to end, as a decode server runs it: the weights (B,
    sB) stay resident in HBM; every step copies the batch's activation rows,
    their scales and the row counts from pinned host memory -- packed in one
    staging buffer, so one host->device copy per step -- launches through the
    public API and copies every group's output back."""
    import torch

    import workloads
    p = workloads.make("c3", seed=0, device="cpu")
    dB = [b.to(dev) for b in p.B]
    dsB = [s.to(dev) for s in p.sB]
    Ms_host = torch.tensor(p.Ms, dtype=torch.int32)
    # one pinned staging buffer holding A, every group's sA and the row counts
    # (each piece 16-byte aligned), mirrored by one device buffer
    pieces = [p.A.contiguous().view(torch.uint8).flatten()] + [s.contiguous().view(torch.uint8).flatten() for s in p.sA] + \
             [Ms_host.view(torch.uint8)]
    offs, total_bytes = [], 0
    for t in pieces:
        offs.append(total_bytes)
        total_bytes += (t.numel() + 15) // 16 * 16
    hpack = torch.zeros(total_bytes, dtype=torch.uint8).pin_memory()
    for o, t in zip(offs, pieces):
        hpack[o:o + t.numel()].copy_(t)
    dpack = torch.empty(total_bytes, dtype=torch.uint8, device=dev)

    def view(i, like):
        n = like.numel() * like.element_size()
        return dpack[offs[i]:offs[i] + n].view(like.dtype).view(like.shape)
    dA = view(0, p.A)
    dsA = [view(1 + g, s) for g, s in enumerate(p.sA)]
    dMs = view(1 + len(p.sA), Ms_host)
    total = sum(p.Ms)
    dC = torch.empty(total, p.N, dtype=torch.bfloat16, device=dev)
    hC = torch.empty(total, p.N, dtype=torch.bfloat16).pin_memory()
    groups = bs.group_descs([(dA[o:o + m], sa, b, sb, dC[o:o + m]) for o, m, sa, b, sb in
                             zip(p.offsets, p.Ms, dsA, dB, dsB)])
    stream = torch.cuda.current_stream(dev)

    def step():
        dpack.copy_(hpack, non_blocking=True)
        bs.fp8_gemm_grouped(groups, dMs, p.N, p.K, stream=stream)
        hC.copy_(dC, non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    ms = t0.elapsed_time(t1) / steps
    h2d = total_bytes
    d2h = 2 * hC.numel()
    return {"value": round(p.algorithmic_bytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "how": "weights resident in HBM; per step the activation rows, their scales and the row "
                   "counts host->device (pinned, packed in one staging buffer: one copy), one grouped "
                   "launch through the public API with a "
                   "prebuilt descriptor array, all outputs device->host"}


def cpu_baseline_sample(name, seconds=15.0):
    """The oracle, as it is, on a bounded sample of the workload's outputs."""
    import numpy as np

    import oracle
    import workloads
    p = workloads.make(name, seed=0, device="cpu")
    A, sA, B, sB = (t.numpy() for t in (p.A, p.sA, p.B, p.sB))
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(0)
    n = 256
    spent, done = 0.0, 0
    t_start = time.perf_counter()
    while spent < seconds:
        ms = rng.integers(0, p.M, n)
        ns = rng.integers(0, p.N, n)
        t0 = time.perf_counter()
        oracle.gemm_sampled(A, sA, B, sB, p.M, p.N, p.K, ms, ns, nthreads=cores)
        spent += time.perf_counter() - t0
        done += n
        if spent < 0.5 * seconds:
            n *= 2
        if time.perf_counter() - t_start > 3 * seconds:
            break
    tflops = 2.0 * p.K * done / spent / 1e12
    return {"value": tflops, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} random output elements of {name} ({p.M}x{p.N}x{p.K}), "
                      f"{spent:.1f} s, fp64 oracle on all host threads"}


def oracle_timings():
    """The oracle on the other workloads: c0, c1 and the grouped decode in
    full on all host threads, the 8192^3 arbitrary-scale GEMM on its first
    512 rows (all columns), and one thread on c0 in full and on the first 128
    rows of c1.  Seconds and effective GFLOP/s of each run."""
    import oracle
    import workloads
    cores = os.cpu_count() or 1
    out = {}

    def timed(key, fn, flops, threads, sample):
        t0 = time.perf_counter()
        fn()
        dt = time.perf_counter() - t0
        out[key] = {"seconds": round(dt, 3), "gflops": round(flops / dt / 1e9, 2), "threads": threads,
                    "sample": sample}

    for name in ("c0", "c1"):
        p = workloads.make(name, seed=0, device="cpu")
        A, sA, B, sB = (t.numpy() for t in (p.A, p.sA, p.B, p.sB))
        timed(name, lambda: oracle.gemm(A, sA, B, sB, p.M, p.N, p.K, nthreads=cores), p.flops, cores,
              f"full {p.M}x{p.N}x{p.K}")
        rows = p.M if name == "c0" else 128
        timed(f"{name}_1thread",
              lambda: oracle.gemm(A[:rows], sA[:(rows + 31) // 32], B, sB, rows, p.N, p.K, nthreads=1),
              2 * rows * p.N * p.K, 1, f"first {rows} rows x all {p.N} columns")
    gp = workloads.make("c3", seed=0, device="cpu")
    timed("c3", lambda: oracle.grouped([gp.A_group(g).numpy() for g in range(gp.G)],
                                       [s.numpy() for s in gp.sA], [b.numpy() for b in gp.B],
                                       [s.numpy() for s in gp.sB], gp.Ms, gp.N, gp.K, nthreads=cores),
          gp.flops, cores, f"full: G={gp.G}, sum M_g={sum(gp.Ms)}, N={gp.N}, K={gp.K}")
    p = workloads.make("c4", seed=0, device="cpu")
    rows = 512
    A, sA, B, sB = (t.numpy() for t in (p.A, p.sA, p.B, p.sB))
    timed("c4", lambda: oracle.gemm(A[:rows], sA[:rows // 32], B, sB, rows, p.N, p.K, nthreads=cores),
          2 * rows * p.N * p.K, cores, f"first {rows} rows x all {p.N} columns of {p.M}x{p.N}x{p.K}")
    return out


def run_ours(args):
    import torch

    import block_scaled_fp8_sm_gb300 as bs
    from block_scaled_fp8_sm_gb300 import build
    world, rank, local = dist_init()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0:
        build.build()
    barrier(world)
    bs.library()
    pk, pk_src = peaks()
    fp8_peak = pk["bf16_tflops"] * FP8_PER_BF16
    hbm_peak = pk["hbm_gbs"]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    results = {}
    hashes = {}
    names = [HEADLINE] + ([] if args.headline_only else ["c1", "c3", "c4", "c4p", "q8", "r1", "f1", "p1", "p1n", "p1e",
                                                         "qo"])
    if args.only:
        names = [args.only]
    launches = 0
    with ClockSampler(local) as clk:
        for name in names:
            run, flops, nbytes, bufs = make_runner(name, dev, bs)
            if not args.only and name != "c4p":
                hashes[name] = {k: sha256_of(v) for k, v in bufs.items()}
            ms = time_device(run, args.steps, args.warmup, dev, flush, world,
                             flush=None if name in UNFLUSHED else "write")
            launches += args.steps
            mean_ms = max_over_ranks(sum(ms) / len(ms), world)
            results[name] = {"ms": mean_ms, "flops": flops, "bytes": nbytes,
                             "ms_min": min(ms), "ms_median": statistics.median(ms)}
            if name == "qo" and not args.only:
                # the same work unfused: bf16 GEMM, then the block quantizer (two launches)
                run_c, _, _, _ = make_runner("qo_chain", dev, bs)
                msc = time_device(run_c, args.steps, args.warmup, dev, flush, world, flush="write")
                launches += 2 * args.steps
                results[name]["ms_chain"] = max_over_ranks(sum(msc) / len(msc), world)
                del run_c
            if name in EXTRA_FLUSH and not args.only:
                for how in EXTRA_FLUSH[name]:
                    msf = time_device(run, args.steps, args.warmup, dev, flush, world, flush=how)
                    launches += args.steps
                    results[name][f"ms_{how or 'not'}_flushed"] = max_over_ranks(sum(msf) / len(msf), world)
            del run, bufs
            torch.cuda.empty_cache()
    status = bs.fp8_status_query()
    if status != 0:
        raise RuntimeError(f"device status after the bench: {bs.fp8_strerror(status)}")
    if args.only:
        r = results[args.only]
        if rank == 0:
            print(json.dumps({"only": args.only, "ms_per_step": r["ms"], "ms_min": r["ms_min"],
                              "tflops": r["flops"] / (r["ms"] * 1e-3) / 1e12,
                              "gbs": r["bytes"] / (r["ms"] * 1e-3) / 1e9}))
        return
    e2e_steps = max(3, args.steps // 5)
    e2e = time_e2e(HEADLINE, e2e_steps, args.warmup, dev, bs, world)
    launches += e2e_steps
    graph_c3 = e2e_c3 = None
    if "c3" in names and world == 1:
        graph_c3 = time_graph_grouped(args.steps, args.warmup, dev, bs, flush)
        launches += 3 * args.steps   # host-table replays; device-table replays (two kernels each)
        e2e_c3 = time_e2e_grouped(e2e_steps, args.warmup, dev, bs, world)
        launches += e2e_steps

    if rank != 0:
        return
    h = results[HEADLINE]
    tflops = world * h["flops"] / (h["ms"] * 1e-3) / 1e12

    def roofline(name):
        r = results[name]
        if name in ("c3", "q8"):
            ach = r["bytes"] / (r["ms"] * 1e-3) / 1e9
            return {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(ach / hbm_peak, 4), "traffic": recorded_traffic(name),
                    "peak_source": f"{pk_src} HBM copy bandwidth"}
        ach = r["flops"] / (r["ms"] * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": round(ach, 1), "peak": round(fp8_peak, 1),
                "unit": "TFLOP/s", "frac": round(ach / fp8_peak, 4),
                "frac_of_nominal_4500": round(ach / 4500.0, 4),
                "traffic": recorded_traffic(name),
                "peak_source": f"{pk_src} bf16 burst x {FP8_PER_BF16} (nominal fp8/bf16 ratio)"}

    extra = {}
    for name in names[1:]:
        r = results[name]
        entry = {"workload": WORKLOAD_NAMES[name], "ms_per_step": round(r["ms"], 4),
                 "roofline": roofline(name)}
        if name in ("c3", "q8"):
            entry["value"] = round(r["bytes"] / (r["ms"] * 1e-3) / 1e9, 1)
            entry["unit"] = "GB/s"
            entry["algorithmic_bytes"] = r["bytes"]
            if name == "c3" and graph_c3:
                entry["graph_replay"] = graph_c3
            if name == "c3" and e2e_c3:
                entry["e2e"] = e2e_c3
            if name in UNFLUSHED:
                entry["l2"] = UNFLUSHED[name]
            else:
                entry["l2"] = "flushed by a 512 MiB write before each launch"
            for how in EXTRA_FLUSH.get(name, ()):
                k = f"ms_{how or 'not'}_flushed"
                if k in r:
                    label = "without_l2_flush" if how is None else f"with_l2_{how}_flush"
                    entry[label] = {"ms_per_step": round(r[k], 4),
                                    "value": round(r["bytes"] / (r[k] * 1e-3) / 1e9, 1), "unit": "GB/s"}
        else:
            entry["value"] = round(r["flops"] / (r["ms"] * 1e-3) / 1e12, 1)
            entry["unit"] = "TFLOP/s"
            if "ms_chain" in r:
                entry["unfused_chain"] = {"ms_per_step": round(r["ms_chain"], 4),
                                          "value": round(r["flops"] / (r["ms_chain"] * 1e-3) / 1e12, 1),
                                          "unit": "TFLOP/s",
                                          "how": "fp8_gemm_blockscaled (bf16 out) then fp8_quantize_blocks"}
        extra[name] = entry

    line = {
        "metric": "block-scaled FP8 GEMM TFLOPS (% FP8 peak); grouped decode GB/s (% HBM)",
        "value": round(tflops, 1),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(h["ms"], 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> f32 accumulate -> bf16",
        "data": "synthetic (seeded; shapes and value distributions of the workloads)",
        "config": {"workload": WORKLOAD_NAMES[HEADLINE], **HEADLINE_SHAPE,
                   "l2": "flushed between timed steps (512 MiB write)",
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline(HEADLINE),
        # launches of this library's kernels inside timed regions: every timed
        # step of every workload (the grouped decode three times: unflushed,
        # read- and write-flushed), its graph replays and the end-to-end steps
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "inputs": {"torch": torch.__version__, "sha256": hashes},
        "extra": extra,
    }
    if e2e:
        ms_e2e, fl, h2d, d2h = e2e
        line["e2e"] = {"value": round(world * fl / (ms_e2e * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": round(ms_e2e, 4),
                       "how": "pinned host buffers; per step all inputs host->device, GEMM, all of C "
                              "device->host; steps pipelined over 3 streams, device buffers doubled"}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_sample(HEADLINE, seconds=args.cpu_seconds)
        line["cpu_baseline"]["other_workloads"] = oracle_timings()
    print(json.dumps(line))


def run_reference(args):
    """The CPU oracle as the reference arm, on rank 0 only."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np

    import oracle
    import workloads
    p = workloads.make(HEADLINE, seed=0, device="cpu")
    A, sA, B, sB = (t.numpy() for t in (p.A, p.sA, p.B, p.sB))
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(1)
    n = args.ref_elements

    def step():
        ms = rng.integers(0, p.M, n)
        ns = rng.integers(0, p.N, n)
        oracle.gemm_sampled(A, sA, B, sB, p.M, p.N, p.K, ms, ns, nthreads=cores)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    tflops = 2.0 * p.K * n / dt / 1e12
    sample = f"{n} random output elements of {HEADLINE} per step ({p.M}x{p.N}x{p.K})"
    line = {
        "impl": "reference",
        "metric": "block-scaled FP8 GEMM TFLOPS (% FP8 peak); grouped decode GB/s (% HBM)",
        "value": tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD_NAMES[HEADLINE], **HEADLINE_SHAPE,
                   "l2": "flushed between timed steps (512 MiB write)",
                   "parallelism": f"replicas x{world}"},
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-elements", type=int, default=65536)
    ap.add_argument("--only", choices=["c1", "c2", "c3", "c4", "c4p", "q8", "r1", "f1", "p1", "p1n", "p1e", "qo"],
                    default=None,
                    help="time one workload only (no e2e, no CPU baseline): profiling runs")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
