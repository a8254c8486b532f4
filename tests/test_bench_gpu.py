"""bench.py's GPU arm on a small case: one JSON line with the fields of the
benchmark contract, values in their plausible ranges (the roofline fraction
against the measured peak, the end-to-end schedules, the clock record)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_bench_line_has_the_contract_fields():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--tokens", "16384", "--steps", "3", "--warmup", "3",
           "--no-cpu-baseline", "--no-split-kv", "--no-masks", "--no-decode", "--no-more-configs",
           "--sustained-s", "0.5"]
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "cpu_baseline",
                "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["data"] == "synthetic" and d["dtype"] == "bf16"
    assert d["config"]["workload"].startswith("llama8b_chunk_16k")
    assert d["value"] > 0 and d["ms_per_step"] > 0
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s"
    assert 0.0 < rf["frac"] < 1.5 and abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    peaks = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks):
        with open(peaks) as f:
            assert rf["peak"] == pytest.approx(float(json.load(f)["bf16_tflops"]))
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    # copies are inside the region: never faster than the device-only step, and the
    # overlapped schedule is no slower than the serial one beyond noise
    assert e2e["ms_per_step"] >= 0.9 * d["ms_per_step"]
    assert e2e["ms_per_step"] <= 1.1 * e2e["serial_ms_per_step"]
    # out: O (bf16), LSE, dQ, dK, dV; in: Q, K, V, dO -- the outputs carry LSE on top
    assert e2e["d2h_bytes_per_step"] == e2e["h2d_bytes_per_step"] + 16384 * 32 * 4
    sus = d["sustained"]
    assert sus["steps"] >= 3 and sus["value"] > 0 and sus["seconds"] >= 0.4
    assert sum(sus["clocks"]["sm_mhz_bins"].values()) == sus["clocks"]["samples"]
    assert d["gpu_launches"] > 0
    assert d["clocks"]["samples"] >= 1 and d["clocks"]["sm_max_mhz"] > 0
    assert d["cpu_baseline"] is None  # skipped here by --no-cpu-baseline
    assert d["pct_of_peak"]["burst"] == pytest.approx(100.0 * d["value"] / rf["peak"])
