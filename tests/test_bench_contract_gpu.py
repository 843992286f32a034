"""The benchmark's result line from a short run of bench.py on the GPU: one JSON
line carrying every key of the measurement contract, with values that agree with
each other (throughput with the step time, the roofline fraction with its parts,
the launch count with the steps, the end-to-end copies declared)."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STEPS, WARMUP = 6, 3


@pytest.fixture(scope="module")
def line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", str(STEPS), "--warmup",
           str(WARMUP), "--no-extras", "--no-cpu-baseline"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    return json.loads(lines[0])


def test_top_level_keys(line):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
              "e2e", "gpu_launches", "clocks"):
        assert k in line, k
    assert isinstance(line["metric"], str) and line["metric"]
    assert (line["n_gpus"], line["steps"], line["warmup"]) == (1, STEPS, WARMUP)
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["vs_baseline"] is None
    assert "workload" in line["config"] and line["data"].startswith("synthetic")
    # the step's four launches (fp16 GEMM, conv, int8 pre-pass, int8 GEMM) per timed step
    assert line["gpu_launches"] == 4 * STEPS


def test_value_is_the_step_rate(line):
    ops = line["config"]["ops_per_step"]
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["value"] == pytest.approx(ops / (line["ms_per_step"] * 1e-3) / 1e12, rel=1e-6)
    per = line["per_shape"]
    parts = sum(v["ms"] for v in per.values())
    # the segments tile the step (events between the calls)
    assert parts == pytest.approx(line["ms_per_step"], rel=0.05)


def test_roofline_fields(line):
    rf = line["roofline"]
    assert rf["bound"] in ("tensor", "hbm", "alu")
    assert rf["unit"] in ("TFLOP/s", "GB/s")
    assert rf["achieved"] > 0 and rf["peak"] > 0
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"], rel=1e-9)
    assert rf["traffic"] is None or rf["traffic"] > 0
    # the dominant kernel's achieved rate is the int8 GEMM kernel's, from its own segment
    k = line["per_shape"]["gemm_s8_zp_8192^3"]
    assert rf["achieved"] == pytest.approx(k["gemm_kernel_tops"], rel=1e-6)


def test_end_to_end_declares_its_copies(line):
    e = line["e2e"]
    assert e["unit"] == line["unit"] and e["value"] > 0
    assert e["h2d_bytes_per_step"] > 200e6 and e["d2h_bytes_per_step"] > 100e6
    # copies of the inputs and outputs inside the timed region cost time
    assert e["value"] < line["value"]


def test_clocks_record(line):
    clk = line["clocks"]
    if clk is None:   # a timed region shorter than the sampler's period
        pytest.skip("no clock sample inside a six-step run")
    assert clk["sm_max_mhz"] > 0 and clk["sm_mhz"] > 0
    assert isinstance(clk["reasons"], list)
