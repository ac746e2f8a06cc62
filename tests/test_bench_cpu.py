"""Host logic of bench.py without a GPU: the reference arm's JSON line, the
silent non-zero ranks, the max-over-ranks timing on 2 gloo ranks, the DRAM
traffic taken only for the sources it was measured on, and the clock record's
summary."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["metric"] == bench.METRIC


def test_reference_arm_other_ranks_exit_silently():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 * (rank + 1), world)
        q.put((rank, got, bench.rank_seed(rank)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(r[1] for r in res) == [20.0, 20.0]
    assert len({r[2] for r in res}) == 2, "ranks must draw distinct buckets"


def test_single_rank_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_traffic_is_used_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    csrc = tmp_path / "lossless_bf16_tensor_zipccl_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("__global__ void k() {}\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.sources_sha()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"k": {"dram_bytes_per_launch": 1234, "sources_sha": sha}}))
    assert bench.traffic_for("k") == 1234
    assert bench.traffic_for("other") is None
    (csrc / "k.cu").write_text("__global__ void k() { }\n")  # the kernel changed since the capture
    assert bench.traffic_for("k") is None


def test_clock_record_summary(tmp_path):
    c = bench.ClockSampler(0)
    c.path = str(tmp_path / "clocks.csv")
    c.proc = object()  # a record exists
    rows = [
        "0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1400.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    (tmp_path / "clocks.csv").write_text("\n".join(rows) + "\n")
    s = c.summary()
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    rows[0] = "0, 1500, 2070, 900.5, 0x40, Not Active, Active, Not Active, Not Active"
    (tmp_path / "clocks.csv").write_text("\n".join(rows) + "\n")
    assert bench.ClockSampler.summary(c)["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert c.lines() == 3
