"""The benchmark's command-line contract, checked without a GPU.

`bench.py --impl reference` times the fp64 oracle on the host's cores over a
bounded sample of the llama7b workload and prints one JSON line with the same
metric, unit and keys as the GPU arm; the GPU arm itself must fail loudly, not
fall back to the CPU, when no GPU is present.
"""

import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, timeout=300):
    return subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True,
                          text=True, timeout=timeout)


def test_reference_arm_prints_one_json_line_with_the_contract_keys():
    res = _run("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"].startswith("fused GEMM-Res-RMSNorm-GEMM TFLOP/s")
    assert d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["dtype"] == "f64" and d["data"] == "synthetic" and d["vs_baseline"] is None
    assert d["ms_per_step"] > 0
    assert "llama7b" in d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == "TFLOP/s"
    assert cb["cores"] >= 1 and "rows per step" in cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_gpu_arm_fails_loudly_without_a_gpu():
    res = _run("--steps", "3", "--warmup", "3", "--extras", "none", "--no-cpu-baseline")
    assert res.returncode != 0
    assert not any(ln.startswith("{") for ln in res.stdout.splitlines())


@pytest.mark.gpu
def test_gpu_arm_prints_the_contract_line():
    """A short GPU run: one JSON line with the roofline, the clocks, the end-to-end
    figure with its copy volumes and the launch count."""
    res = _run("--steps", "3", "--warmup", "3", "--extras", "none", "--no-cpu-baseline", timeout=900)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    assert d["unit"] == "TFLOP/s" and d["value"] > 0 and d["steps"] == 3 and d["warmup"] == 3
    assert d["dtype"] == "bf16" and d["scaling"] == "weak" and d["higher_is_better"] is True
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 4 * 3  # fwd (3 launches) + dgrad (1) per timed step
