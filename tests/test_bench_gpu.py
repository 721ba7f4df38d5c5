"""bench.py's output contract on a GPU: one JSON line with the keys the measurement needs.

Runs the bench on the small tiny workload (a few seconds) as a separate process, the way it
is run for the record, and checks the line's fields and their consistency: the throughput
and its step time, the roofline block, the end-to-end block with its copied bytes, the
launch count and the clock record sampled inside the timed region.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def run_bench(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-3000:]
    return json.loads(lines[0])


def test_bench_line_on_the_tiny_workload():
    steps = 4
    d = run_bench("--workload", "tiny", "--steps", str(steps), "--warmup", "3",
                  "--no-workloads", "--no-cpu-baseline")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == 3
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0
    # value is the step's FLOPs (fused pass + chunk path, 4*B*H*N^2*D each) over its time
    B, H, N, D = (d["config"][k] for k in ("B", "H", "N", "D"))
    flops = 2 * 4 * B * H * N * N * D
    assert d["value"] == pytest.approx(flops / (d["ms_per_step"] * 1e-3) / 1e12, rel=1e-6)
    assert d["config"]["workload"].startswith("tiny")
    roof = d["roofline"]
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    assert roof["achieved"] > 0 and roof["peak"] > 0
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"], rel=1e-9)
    e2e = d["e2e"]
    assert e2e["unit"] == d["unit"] and e2e["value"] > 0
    # per step: Q, K, V uploaded (bf16); both outputs (fp32 O and LSE) downloaded
    assert e2e["h2d_bytes_per_step"] == 3 * B * H * N * D * 2
    assert e2e["d2h_bytes_per_step"] == 2 * (B * H * N * D * 4 + B * H * N * 4)
    assert e2e["fused_bitwise_equal_to_device"] is True
    assert d["gpu_launches"] == 3 * steps  # fused pass, chunk launch, merge per step
    clk = d["clocks"]
    assert clk["samples"] >= 1 and clk["sm_max_mhz"] > 0
    assert clk["sm_min_mhz"] <= clk["sm_mhz"] <= clk["sm_max_mhz"]
    assert "timed region" in clk["sampling"]


def test_profile_case_runs_silently():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny",
                          "--profile-case", "fused", "--steps", "1", "--warmup", "3"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    assert not [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
