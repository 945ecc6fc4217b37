"""bench.py's host-side contract, on the CPU: the reference arm's JSON line and
the traffic record's source check."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "A",
                          "--steps", "2", "--warmup", "1"], cwd=ROOT, capture_output=True,
                         text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("A:")


def test_traffic_record_requires_matching_source(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    rec = bench.traffic_record()
    if rec is not None:                      # the committed record matches the sources
        assert float(rec["dram_bytes_per_launch_full"]) > 0
    monkeypatch.setattr(bench, "gemm_source_sha", lambda: "0" * 64)
    assert bench.traffic_record() is None    # any other source revision: no traffic claim
