"""Host-side logic of bench.py, on CPU: the multi-rank aggregation (gloo,
world size 2), the clock-sample parser, the byte counts and the reference
arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from speculative_decoding_tree_hybrid_gb300 import workloads as wl  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r processed 10 units in r+1 seconds: the job rate is 2*10 / 2 s
    value, t = bench.aggregate(10.0, float(rank + 1), dist)
    bench.barrier(dist)
    q.put((rank, value, t))
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, value, t in res:
        assert t == 2.0 and value == pytest.approx(10.0)


def test_aggregate_single_process():
    v, t = bench.aggregate(6.0, 3.0, None)
    assert v == 2.0 and t == 3.0


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
