"""The bench's own line on the GPU, a short run without the extra workloads and
the CPU baseline: one JSON line with the fields the line promises, a roofline
whose fraction is its achieved rate over its peak, an end-to-end figure from
three timed loops that does not beat the device-resident one, sampled clocks
and a count of the library's launches."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_on_the_gpu():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3", "--no-extra",
                        "--no-cpu-baseline"], capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "clocks", "gpu_launches"):
        assert key in d, key
    assert d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True and d["value"] > 0
    assert "workload" in d["config"]
    # the step is a forward and a backward: value is their time's rate, ms_per_step their sum
    assert d["ms_per_step"] > 0

    rf = d["roofline"]
    assert rf["bound"] in ("tensor", "hbm") and rf["unit"] in ("TFLOP/s", "GB/s")
    assert rf["achieved"] > 0 and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert rf["traffic"] is None or rf["traffic"] > 0

    e = d["e2e"]
    assert e["unit"] == d["unit"] and e["value"] > 0
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    loops = e["loops_ms_per_step"]
    assert len(loops) == 3 and all(t > 0 for t in loops)
    assert abs(e["ms_per_step"] - sorted(loops)[1]) < 1e-3  # the median loop
    assert e["value"] <= d["value"] * 1.02  # host copies inside the timed region cannot make it faster
    assert e["link"]["copy_bound_tflops"] > 0

    c = d["clocks"]
    assert c["sm_max_mhz"] > 0 and "reasons" in c
    assert d["gpu_launches"] == 3 * 4  # fa_fwd and the backward's pre, main and post kernels per step
