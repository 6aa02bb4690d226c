"""Host-side parts of bench.py (CPU only): the reference arm's JSON line,
the rule that a committed DRAM-traffic figure is used only while the
row-statistics sources are unchanged, and the whole-job rate."""

import importlib.util
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_reference_arm_prints_one_contract_line():
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "4", "--warmup", "1"], capture_output=True, text=True, env=env,
                         cwd=ROOT, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 4 and d["warmup"] == 1
    assert d["metric"] == "verified draft positions/sec" and d["unit"] == "positions/s"
    assert d["higher_is_better"] is True and d["value"] > 0
    cb = d["cpu_baseline"]
    bench = _bench()
    assert cb["kind"] == "oracle" and cb["cores"] == bench.host_cores() and cb["value"] == d["value"]
    assert cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "batch64-bf16"


def test_traffic_figure_only_while_sources_hash_the_same(monkeypatch):
    bench = _bench()
    with open(bench.TRAFFIC) as f:
        record = json.load(f)
    if record["csrc_hash"] == bench.csrc_hash():
        assert bench.traffic_per_launch() == record["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "csrc_hash", lambda *a, **k: "0" * 16)
    assert bench.traffic_per_launch() is None


def test_whole_job_rate_counts_every_rank():
    bench = _bench()
    # 448 positions per rank-step, 100 steps, 2 ranks, slowest rank 5 ms
    assert bench.whole_job_rate(448, 100, 2, 5.0) == 448 * 100 * 2 / 0.005


def test_oracle_host_times_one_thread_and_every_core():
    """The oracle timing of the cpu_baseline and per-config keys: a saved
    workload, one thread here, then a spawned process per core."""
    sys.path.insert(0, ROOT)
    import bench  # importable by name, so the spawned workers find its functions
    from speculative_decoding_verification_73_gb300 import workloads
    host = bench.OracleHost()
    try:
        host.start()
        out = host.time_requests("tiny-f32", workloads.tiny_f32(), budget_s=0.3)
    finally:
        host.close()
    assert out["cores"] == bench.host_cores() and out["value"] > 0 and out["unit"] == bench.UNIT
    assert out["single_thread"]["cores"] == 1 and out["single_thread"]["value"] > 0
    assert not os.path.exists(host.dir)
