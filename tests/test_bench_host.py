"""Host-side logic of bench.py, on CPU: the single-GPU guard (a run asked
for more GPUs prints one skip line and does no GPU work), the clock-sample
parser, the byte counts and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from speculative_decoding_tree_hybrid_gb300 import workloads as wl  # noqa: E402


def test_throughput():
    v, t = bench.throughput(6.0, 3.0)
    assert v == 2.0 and t == 3.0


@pytest.mark.parametrize("env,args", [({"WORLD_SIZE": "2", "RANK": "0"}, []), ({}, ["--gpus", "4"])])
def test_multi_gpu_run_prints_one_skip_line(env, args):
    """More than one GPU: no GPU work, one JSON line with the reason (rank 0)."""
    e = dict(os.environ, **env)
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args, "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=120, cwd=ROOT, env=e)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["skipped"] and line["value"] is None and line["n_gpus"] > 1


def test_multi_gpu_other_ranks_print_nothing():
    e = dict(os.environ, WORLD_SIZE="2", RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=120, cwd=ROOT, env=e)
    assert out.returncode == 0, out.stderr
    assert not [l for l in out.stdout.splitlines() if l.startswith("{")]


def test_cpu_model_is_named():
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()


def test_clock_summary_parser():
    c = bench.ClockSampler(0)
    c.lines = ["0, 1900, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Active",
               "0, 1950, 2070, 910.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 1800, 2070, 905.0, 0x0, Active, Not Active, Not Active, Not Active",
               "garbage"]
    s = c.summary()
    assert s["sm_mhz"] == 1900 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert bench.ClockSampler(0).summary()["samples"] == 0


def test_kv_bytes_of_llama_config():
    cfg = wl.CONFIGS["llama8b"]
    inp = wl.Inputs(cfg, None, None, None, wl.cache_lengths(cfg), None, None, None)
    assert bench.kv_bytes(inp) == 134217728
    assert bench.all_bytes(inp) > bench.kv_bytes(inp)


def test_traffic_record_requires_current_sources(tmp_path, monkeypatch):
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps({"llama8b": {"k": {"source_hash": "stale", "dram_bytes_per_launch": 1.0}}}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("llama8b", "k") is None
    f.write_text(json.dumps({"llama8b": {"k": {"source_hash": bench.kernel_source_hash(),
                                               "dram_bytes_per_launch": 5.0}}}))
    assert bench.recorded_traffic("llama8b", "k") == 5.0
    assert bench.recorded_traffic("llama8b", "other") is None


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--steps", "2", "--warmup", "1", "--ref-rows", "8"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_kv_layout_option():
    assert bench.parse_kv_layout("hnd") == ("hnd", 0)
    assert bench.parse_kv_layout("nhd") == ("nhd", 0)
    assert bench.parse_kv_layout("nhd:16") == ("nhd", 16)
    assert bench.parse_kv_layout("hnd:256") == ("hnd", 256)
    with pytest.raises(SystemExit):
        bench.parse_kv_layout("bshd")
