"""The bench's JSON contract on the CPU: the reference arm (the oracle timed on
the host) on the small 1024x1024 workload prints one well-formed line, and the
byte accounting and the traffic lookup behave as documented."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "1d_1024x1024_bf16", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] >= 3
    assert d["config"]["workload"] == "1d_1024x1024_bf16"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"] and "rows" in cb["sample"]
    assert cb.get("host_cores", 0) >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_workload_bytes_follow_the_stated_accounting():
    import bench
    from nvfp4_block_scaled_amax_gb300 import inputs
    # BF16 row+col: 2 bytes in, two directions of codes (0.5 B) and scales (1/16 B) out
    assert bench.workload_bytes(inputs.WORKLOADS["2d_8192x5120_bf16"]) == 8192 * 5120 * 3.125
    # FP32 in: 4 bytes per element instead of 2
    assert bench.workload_bytes(inputs.WORKLOADS["1d_4096x3072_fp32"]) == 4096 * 3072 * 5.125
    # row-scaled: one direction, plus one FP32 amax per row
    spec = inputs.WORKLOADS["rowscaled_16384x4096_bf16"]
    assert bench.workload_bytes(spec) == pytest.approx(16384 * 4096 * (2 + 0.5 + 1 / 16) + 16384 * 4)


def test_traffic_is_reported_only_for_current_sources(monkeypatch):
    import bench
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    for name, e in d.items():
        # the committed entry is reported while it matches the current sources of its kernel
        cur = bench.kernel_source_hash(e["source"])
        assert bench.ncu_traffic(name) == (e["dram_bytes_per_call"] if cur == e["kernel_hash"] else None)
    # once the kernel's sources change, the figure is unknown
    monkeypatch.setattr(bench, "kernel_source_hash", lambda source: "0" * 16)
    for name in d:
        assert bench.ncu_traffic(name) is None
    # the headline's figure is current
    monkeypatch.undo()
    assert bench.ncu_traffic("2d_8192x5120_bf16") is not None
