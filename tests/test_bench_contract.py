"""bench.py's output contract: one JSON line with the keys and types the measurement needs.
The reference arm (the CPU oracle timed on a bounded sample) runs without a GPU; the dense
line is checked on a GPU with a short run."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout):
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def _common(line, steps):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e"):
        assert key in line, key
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["steps"] == steps and line["warmup"] >= 3 and line["vs_baseline"] is None
    assert "workload" in line["config"] and "model" not in line["config"]
    e2e = line["e2e"]
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert key in e2e, key


def test_reference_arm_line():
    line = _run(["--impl", "reference", "--steps", "2", "--warmup", "3"], timeout=600)
    _common(line, 2)
    assert line["impl"] == "reference" and line["dtype"] == "f64"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == pytest.approx(line["value"])
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_dense_line():
    steps = 4
    line = _run(["--steps", str(steps), "--warmup", "3"], timeout=900)
    _common(line, steps)
    assert line["n_gpus"] == 1 and line["scaling"] == "weak" and line["dtype"] == "e4m3"
    assert line["gpu_launches"] == 20 * steps
    roof = line["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in roof, key
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    clk = line["clocks"]
    for key in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert key in clk, key
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] > 0 and line["e2e"]["d2h_bytes_per_step"] > 0
    assert line["quantize"]["GB/s"] > 0 and line["gemm"]["TFLOP/s"] > 0
    rq = line["roofline_quantize"]
    assert rq["bound"] == "hbm" and rq["unit"] == "GB/s"
    assert rq["frac"] == pytest.approx(rq["achieved"] / rq["peak"])
    sec = line["secondary"]
    moe = sec["moe_qwen3_30b_a3b"]
    for proj in ("gate_up", "down"):
        for op in ("fprop", "dgrad", "wgrad"):
            assert moe[proj][op]["TFLOP/s"] > 0 and moe[proj][op]["frac_of_roof"] > 0
    assert sec["weight_sync_qwen3_8b"]["weights"] == 144
    assert [r["tokens"] for r in sec["microbatch_sweep"]] == [1024, 2048, 4096, 4608, 8192, 16384]
