"""bench.py prints one JSON line with the keys its consumers read.

The reference arm (the oracle on host cores) runs here on CPU; the GPU arm
(forward and backward passes, kernel-only and end to end) runs on a GB300.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
             "vs_baseline", "dtype", "data", "config", "e2e"}


def run_bench(*args, timeout=900):
    out = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True, text=True,
                         timeout=timeout, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out
    return json.loads(lines[0])


def test_reference_arm_line():
    d = run_bench("--impl", "reference", "--steps", "1", "--warmup", "3", timeout=600)
    assert BASE_KEYS <= set(d) and d["impl"] == "reference"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["value"] > 0 and d["config"]["workload"] == "b8h32n4096d128_bf16_qk3"


@pytest.mark.gpu
@pytest.mark.parametrize("args", [[], ["--pass", "bwd"]], ids=["fwd", "bwd"])
def test_gpu_arm_line(args):
    d = run_bench(*args, "--steps", "4", "--warmup", "3", "--no-cpu-baseline")
    assert BASE_KEYS <= set(d)
    assert d["n_gpus"] == 1 and d["steps"] == 4 and d["warmup"] >= 3 and d["higher_is_better"] is True
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and 0 < r["frac"] < 1.2
    assert abs(r["achieved"] / r["peak"] - r["frac"]) < 1e-3
    assert "traffic" in r
    assert d["gpu_launches"] >= d["steps"]
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    c = d["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(c)
    dist = d["ms_per_step_dist"]
    assert dist["n"] == 4 and dist["p10"] <= dist["median"] <= dist["p90"]
    assert d["config"]["l2"]


@pytest.mark.gpu
def test_gpu_arm_line_parity_and_sustained_leg():
    """The forward line carries the parity figures of the timed output on the
    heads the CPU baseline computed, and the seconds-long sustained leg."""
    d = run_bench("--workload", "b8h12n2048d128_f16", "--steps", "4", "--warmup", "3", "--no-e2e",
                  "--cpu-seconds", "2", "--sustained-seconds", "0.5")
    p = d["parity"]
    assert p["ok"] and p["heads"] >= 1 and p["cos"] >= 0.999 and p["max_abs"] <= 1e-2
    s = d["sustained"]
    assert s["steps"] >= 10 and s["value"] > 0 and abs(s["value"] / s["peak"] - s["frac"]) < 1e-3
    assert {"sm_mhz", "reasons"} <= set(s["clocks"])
    assert 0 < d["pct_of_measured_peak"] and 0 < d["pct_of_datasheet_peak"] < d["pct_of_measured_peak"]
