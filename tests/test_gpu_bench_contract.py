"""The benchmark's one-line JSON report on the GPU: a short run of `bench.py` as a user (or the
round-end harness) would start it, checked field by field against the report's contract."""
import json
import math
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402  (the module's constants only; nothing runs on import)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def report():
    steps, warmup = 3, 3
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", str(steps), "--warmup",
                          str(warmup), "--no-cpu-baseline"], cwd=ROOT, capture_output=True, text=True,
                         timeout=900)
    assert out.returncode == 0, out.stderr[-4000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert lines, out.stdout[-2000:]
    return json.loads(lines[-1]), steps, warmup


def test_headline_fields(report):
    r, steps, warmup = report
    assert r["metric"] == bench.METRIC and r["unit"] == bench.UNIT
    assert r["value"] > 0 and math.isfinite(r["value"])
    assert r["n_gpus"] == 1 and r["steps"] == steps and r["warmup"] == warmup
    assert r["ms_per_step"] > 0 and r["higher_is_better"] is True
    assert r["scaling"] == "weak" and r["vs_baseline"] is None
    assert r["dtype"] == "nvfp4" and r["data"] == "synthetic"
    assert r["config"]["workload"] == bench.WORKLOAD_NAME
    # step rate = the step's GEMM FLOPs over the step time
    flops = 2 * 4608 * (3072 * 9216 + 3072 * 24576 + 12288 * 3072)
    assert r["value"] == pytest.approx(flops / (r["ms_per_step"] * 1e-3) / 1e12, rel=1e-3)
    # six launches a step: one quantize and one GEMM for each of the three linears
    assert r["gpu_launches"] == 6 * steps


def test_roofline_fields(report):
    rf = report[0]["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s"
    assert rf["achieved"] > 0 and rf["peak"] > 0
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"], abs=1e-3)
    assert rf["traffic"] is None or rf["traffic"] > 0
    assert 0 < rf["instruction_ceiling"] and rf["frac_of_instruction_ceiling"] == pytest.approx(
        rf["achieved"] / rf["instruction_ceiling"], abs=1e-3)


def test_breakdown_covers_every_launch_of_the_step(report):
    b = report[0]["breakdown"]
    for name in ("qkv_rmsnorm", "gated_up", "down_bias"):
        assert b[f"gemm_{name}"]["tflops"] > 0 and b[f"quantize_{name}"]["gbs"] > 0
    assert b["quantize_down_bias_static_scale"]["gbs"] > 0


def test_end_to_end_fields(report):
    e = report[0]["e2e"]
    assert e["value"] > 0 and e["unit"] == bench.UNIT
    # bf16 activations in ([4608, 3072] twice, [4608, 12288]) and bf16 outputs back
    assert e["h2d_bytes_per_step"] == 2 * 4608 * (3072 + 3072 + 12288)
    assert e["d2h_bytes_per_step"] == 2 * 4608 * (9216 + 12288 + 3072)
    assert 0 < e["copy_floor"]["frac"] < 1.5


def test_clock_record(report):
    c = report[0]["clocks"]
    assert c["sm_mhz"] > 0 and isinstance(c["reasons"], list)
