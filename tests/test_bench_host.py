"""Host checks of the benchmark script (no device needed): the reference arm
prints one JSON line with every key of the benchmark contract, and each DRAM
traffic figure committed under profiles/ names a kernel the benchmark knows
and was taken on that kernel's current sources (so the headline's
roofline.traffic is reported, not withheld)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert KEYS <= set(d)
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["config"]["workload"] == bench.WORKLOAD["workload"]


def test_committed_traffic_matches_current_sources():
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert "diamond" in d
    for workload, rec in d.items():
        assert rec["kernel"] in bench.KERNEL_SOURCES, workload
        assert rec["sources"] == bench.sources_hash(rec["kernel"]), workload
        assert bench.traffic_for(rec["kernel"], workload) == pytest.approx(rec["dram_bytes_per_launch"])
