"""bench.py's result line on a small corpus: one JSON line carrying every key
the measurement contract asks for, with consistent values (the default run
uses 1M x 1024 and the companion workloads; this one 100k rows and the
single-query path only)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_has_the_contract_keys():
    steps, warmup = 20, 3
    cmd = [sys.executable, "bench.py", "--steps", str(steps), "--warmup", str(warmup), "--n", "100000",
           "--queries", "64", "--no-batched", "--no-int32", "--no-views", "--no-cosine", "--no-sweep"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    rec = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "gpu_launches", "clocks", "device"):
        assert key in rec, key
    assert rec["n_gpus"] == 1 and rec["steps"] == steps and rec["warmup"] == warmup
    assert rec["value"] > 0 and rec["higher_is_better"] is True and rec["scaling"] == "weak"
    assert rec["gpu_launches"] == steps and "workload" in rec["config"]
    assert abs(rec["value"] - 100000 * 1024 * 4 / (rec["ms_per_step"] * 1e-3) / 1e9) <= 0.01 * rec["value"]
    roof = rec["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in roof, key
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    cpu = rec["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] > 0 and cpu["cores"] >= 1 and cpu["sample"]
    assert cpu["one_core"]["value"] > 0
    e2e = rec["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] == 1024 * 4 and e2e["d2h_bytes_per_step"] > 0
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(rec["clocks"])
    assert rec["clocks"]["samples"] >= 1
    assert {"headline.k8", "e2e.k8", "config1.l2", "config1.flushed", "config1.e2e"} <= set(rec["clocks"]["regions"])
    assert rec["device"]["name"]
    c1 = rec["config1"]
    assert c1["queries"] == 16 and c1["oracle_checked_queries"] == 16 and c1["launches_per_call"] == 1
    for key in ("p50_us", "p99_us", "flushed_p50_us", "e2e_p50_us"):
        assert c1[key] > 0, key
    assert rec["per_k"]["8"]["launches_per_step"] == 1
