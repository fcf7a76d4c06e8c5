"""Host-side logic of bench.py: roofline arithmetic, the weak-scaling
aggregate, the max-over-ranks timing reduction on two gloo ranks, and the
reference arm (the oracle) on CPU."""
import json
import os
import subprocess
import sys

import pytest

import bench
from mamba_ssd_chunked_gb300.inputs import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_bytes_and_flops_of_the_headline_workload():
    w = WORKLOADS["mamba2_2p7b_layer"]
    # x + y (2 x 167.8 MB) + B + C (2 x 4.2 MB) + dt (5.2 MB) + init + final (2 x 10.5 MB) + 3 per-head vectors
    assert bench.algorithmic_bytes(w) == 370148288
    assert abs(bench.algorithmic_flops(w) / 1e9 - 64.96) < 0.01


def test_algorithmic_bytes_counts_init_only_when_given():
    w = WORKLOADS["mamba2_130m_layer"]
    x = 8 * 2048 * 24 * 64 * 2
    bc = 8 * 2048 * 128 * 2
    dt = 8 * 2048 * 24 * 4
    fs = 8 * 24 * 64 * 128 * 4
    assert bench.algorithmic_bytes(w) == 2 * x + 2 * bc + dt + fs + 3 * 24 * 4


def test_weak_scaling_aggregate_takes_the_slowest_rank():
    v, t = bench.aggregate([0.002, 0.003], 1000, 2)
    assert t == 0.003 and abs(v - 2 * 1000 / 0.003) < 1e-6


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    m = bench.max_over_ranks(dist, 1.0 + rank)
    out.put((rank, m))
    dist.destroy_process_group()


def test_max_over_ranks_on_two_gloo_ranks():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(timeout=120)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert res == [(0, 2.0), (1, 2.0)]
    assert all(p.exitcode == 0 for p in ps)


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_fp32",
                        "--steps", "2", "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_is_silent_on_other_ranks():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_fp32",
                        "--steps", "1", "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_profiled_traffic_is_dropped_when_the_kernel_changed(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "kernel_source_hash", lambda *a: "not-the-profiled-source")
    assert bench.profiled_traffic("mamba2_2p7b_layer") is None
