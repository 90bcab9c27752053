"""Host-side checks of bench.py: the multi-rank timing reduction (gloo, 2 ranks
on CPU), the throughput aggregation, and the oracle reference arm's JSON line."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench
        # rank r reports prefill 10+r ms, decode 5-r ms: the slowest rank wins per entry
        got = bench.reduce_max([10.0 + rank, 5.0 - rank, 1.5], world, "cpu")
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == out[1] == [11.0, 5.0, 1.5]


def test_aggregate_throughput_is_weak_scaling_sum():
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks, 1e12 FLOP per step each, 10 steps in 20 ms on the slowest rank
    assert bench.aggregate_throughput(1e12, 2, 10, 20.0) == pytest.approx(2 * 1e12 * 10 / 0.02)


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOPS" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_exponential_count_and_nvtx_fallback():
    sys.path.insert(0, ROOT)
    import bench
    # one exponential per attended (query, key) pair
    assert bench.prefill_exps(B=1, Hq=1, N=4, causal=True) == 10
    assert bench.prefill_exps(B=2, Hq=3, N=4, causal=False) == 2 * 3 * 16
    push, pop = bench.nvtx_ranges()
    push("x")
    pop()


def test_traffic_is_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    src = tmp_path / "attention_fa2_fwd_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "k.cuh").write_text("kernel v1\n")
    import hashlib
    sha = hashlib.sha256(b"kernel v1\n").hexdigest()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps({"k": {"source": "k.cuh", "source_sha256": sha,
                                                         "dram_bytes_per_launch": 123}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "PROFILES", str(prof))
    assert bench.profiled_traffic("k") == 123.0
    (src / "k.cuh").write_text("kernel v2\n")  # the source changed after the capture
    assert bench.profiled_traffic("k") is None
    assert bench.profiled_traffic("missing") is None
