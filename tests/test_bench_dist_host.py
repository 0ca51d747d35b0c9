"""The benchmark's multi-rank host logic on CPU: two ranks over gloo (the
GEMM itself runs as independent replicas, so the ranks only meet for the
timing barrier and the max over ranks), and the reference arm, which only
rank 0 runs and prints."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    bench = _bench()
    w, r, _ = bench.dist_init()
    bench.barrier(w)
    m = bench.max_over_ranks(1.5 + rank, w)   # per-rank step times; the slowest rank counts
    out.put((r, w, m))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_ranks_gloo_barrier_and_max():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2, 2.5), (1, 2, 2.5)]


def test_single_rank_needs_no_process_group():
    bench = _bench()
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_on_rank0_only(rank):
    env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--ref-elements", "64"],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if rank != 0:
        assert lines == []
        return
    line = json.loads(lines[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_source_hash_ignores_comments_only():
    bench = _bench()
    code = "int f(int x) {\n    return x + 1;   // one more\n}\n/* block\n comment */\n"
    assert bench._code_only(code) == bench._code_only("int f(int x) {\n    return x + 1;\n}\n")
    assert bench._code_only(code) != bench._code_only("int f(int x) {\n    return x + 2;\n}\n")


def test_traffic_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    bench = _bench()
    rec = {"source_hash": bench.source_hash(), "c1": {"dram_bytes_per_launch": 123, "source_hash": bench.source_hash()},
           "c2": {"dram_bytes_per_launch": 456, "source_hash": "0000000000000000"}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC", str(path))
    assert bench.recorded_traffic("c1") == 123     # captured on this source
    assert bench.recorded_traffic("c2") is None    # another kernel source
    assert bench.recorded_traffic("c3") is None    # never captured

