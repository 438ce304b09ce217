"""The bench's output contract: one JSON line with the keys a driver reads.

The reference arm (the fp64 oracle over all of one sample) runs on the CPU in
well under a minute per step; the library's arm needs a GPU.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


BASE_KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
             "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e")


def _check_common(line, steps, warmup):
    for k in BASE_KEYS:
        assert k in line, k
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["steps"] == steps and line["warmup"] == warmup and line["n_gpus"] == 1
    assert line["scaling"] == "weak" and line["data"] == "synthetic"
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["config"]["workload"] == "up_proj_bf16_B4_T4096_d2048_p8192"
    e2e = line["e2e"]
    assert e2e["unit"] == "tokens/s" and e2e["value"] > 0
    assert e2e["h2d_bytes_per_step"] >= 0 and e2e["d2h_bytes_per_step"] >= 0


def test_reference_arm_line():
    line = _run(["--impl", "reference", "--steps", "1", "--warmup", "1"], timeout=600)
    _check_common(line, 1, 1)
    assert line["impl"] == "reference" and line["dtype"] == "f64"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert "sample" in cb and cb["unit"] == "tokens/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_library_arm_line():
    line = _run(["--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--no-extra"], timeout=900)
    _check_common(line, 3, 3)
    assert "impl" not in line or line["impl"] != "reference"
    assert line["dtype"] == "bf16" and line["gpu_launches"] == 3 * 17
    roof = line["roofline"]
    assert roof["bound"] in ("hbm", "tensor") and roof["unit"] in ("GB/s", "TFLOP/s")
    assert roof["achieved"] > 0 and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    assert set(line["breakdown"]) == {"hutch", "hutchpp", "exact_direct", "exact_ghost",
                                      "clipped_noisy_grad"}
    assert set(line["layer_totals"]) == {"hutch+grad", "hutchpp+grad", "exact_direct+grad",
                                         "exact_ghost+grad"}
    assert "sm_mhz" in line["clocks"] and "reasons" in line["clocks"]
    assert "sm_mhz" in line["clocks_rows"] and "reasons" in line["clocks_rows"]
    # the roofline is the slowest row of the step, as timed inside the step
    bd = line["breakdown"]
    dom = max(bd, key=lambda r: bd[r]["in_step_ms"])
    assert roof["kernel"] == dom and roof["timing"].startswith("inside the step")
    scale = 1e9 if roof["unit"] == "GB/s" else 1e12
    ach = bd[dom]["algorithmic"] / (bd[dom]["in_step_ms"] * 1e-3) / scale
    assert abs(roof["achieved"] - ach) < 1e-3 * ach + 0.01
    # the end-to-end leg moves the inputs in and the results out every step
    assert line["e2e"]["h2d_bytes_per_step"] == 2 * 4 * 4096 * (2048 + 8192)
    assert line["e2e"]["d2h_bytes_per_step"] >= 4 * 2048 * 8192
    # the other standard workloads, each with the rows it names
    cf = line["configs"]
    assert set(cf) == {"tiny_f32_B4_T64_d32_p48", "exact_bf16_B8_T512_d768_p768",
                       "q_proj_bf16_B4_T4096_d2048_p2048", "long_ctx_bf16_B2_T16384_d2048_p2048"}
    assert set(cf["long_ctx_bf16_B2_T16384_d2048_p2048"]["rows"]) == {
        "hutch", "hutchpp", "exact_direct", "clipped_noisy_grad"}
    for name, c in cf.items():
        for r, e in c["rows"].items():
            assert e["ms"] > 0, (name, r)
            if e["bound"] != "latency":
                assert 0 < e["frac"] < 1.5, (name, r)


def test_clock_summary_windows():
    """The clock summary keeps the samples inside a window (else the two
    nearest), reports their median SM clock and every throttle reason seen
    among them."""
    sys.path.insert(0, ROOT)
    import bench
    cs = bench.ClockSampler(0)
    inactive = ["Not Active"] * 5
    capped = ["Active", "Not Active", "Not Active", "Not Active", "Active"]
    cs.rows = [(10.0, 2070.0, 2070.0, inactive), (10.1, 2070.0, 2070.0, inactive),
               (10.2, 2070.0, 2070.0, inactive), (11.0, 1840.0, 2070.0, capped),
               (11.1, 1830.0, 2070.0, capped), (11.2, 2070.0, 2070.0, inactive)]
    step = cs.summary(9.95, 10.25)
    assert step["sm_mhz"] == 2070.0 and step["reasons"] == [] and step["samples_in_window"] == 3
    rows = cs.summary(10.95, 11.25)
    assert rows["sm_mhz"] == 1840.0 and rows["reasons"] == ["sw_power_cap"]
    assert rows["samples_in_window"] == 3
    outside = cs.summary(20.0, 20.5)
    assert outside["samples_in_window"] == 0 and outside["samples"] == 2
    cs.rows = []
    assert cs.summary(0.0, 1.0) is None
