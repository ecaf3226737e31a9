"""The benchmark's JSON line keeps its contract: one line on stdout with the
metric, value and unit, the step timing, the roofline of the dominant
kernel, the clocks seen during the timed region, the end-to-end figure
with its host<->device bytes, the count of library kernel launches and the
CPU oracle baseline.  Run on a small workload so the test stays short."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def _run(*args):
    out = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def _check_line(d, steps, warmup):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup",
              "ms_per_step", "higher_is_better", "scaling", "vs_baseline",
              "dtype", "data", "config", "roofline", "gpu_launches",
              "clocks", "e2e", "cpu_baseline"):
        assert k in d, k
    assert d["steps"] == steps and d["warmup"] == warmup
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["dtype"] == "bf16" and d["data"] == "synthetic"
    assert "workload" in d["config"] and "l2" in d["config"]
    r = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["bound"] == "tensor" and 0 < r["frac"] < 1.5
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    # the tensor core's own rate at the sampled clock bounds every kernel
    assert 0 < r["frac_at_clock"] <= 1.0
    assert abs(r["frac_at_clock"] * r["tensor_peak_at_clock"]
               - r["achieved"]) < 1e-6 * r["achieved"]
    assert d["gpu_launches"] > 0
    c = d["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(c)
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0
    assert e["d2h_bytes_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1
    assert cb["sample"]


def test_bench_line_kv_pages():
    d = _run("--config", "mid", "--steps", "3", "--warmup", "3",
             "--cpu-positions", "2")
    _check_line(d, 3, 3)
    assert d["config"]["workload"] == "mid"
    assert "phases" in d and "side_kernels" in d


def test_bench_line_latent_pages():
    d = _run("--config", "latent_mid", "--steps", "3", "--warmup", "3",
             "--latent-cpu-positions", "1")
    _check_line(d, 3, 3)
    assert d["config"]["workload"] == "latent_mid"
