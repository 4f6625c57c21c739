"""The benchmark's output contract: one JSON line with the metric, the
whole-job value, the roofline of the dominant kernel, the end-to-end number
with its host-device byte counts, the clocks seen and the kernel launch count
(GPU); and the reference line, the CPU oracle on the host cores (no GPU)."""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT


def _line(args, timeout):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_line():
    d = _line(["--impl", "reference", "--steps", "2", "--warmup", "3"], 600)
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["vs_baseline"] is None and d["config"]["workload"].startswith("llama3_8b_decode")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


@pytest.mark.gpu
def test_gpu_bench_line():
    d = _line(["--main-only", "--no-cpu-baseline", "--steps", "10", "--warmup", "3"], 900)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "clocks",
              "gpu_launches"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 10 and d["warmup"] == 3 and d["scaling"] == "weak"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["gpu_launches"] > 0
    assert "workload" in d["config"] and "l2" in d["config"]
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["achieved"] == d["value"]
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == "GB/s"
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
