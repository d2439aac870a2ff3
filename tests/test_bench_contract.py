"""bench.py's output contract: one JSON line with the keys its readers use.

The reference arm (the fp64 oracle on the host cores) runs on the CPU; our arm
needs the GPU.  Both run bench.py as a subprocess, as it is launched for real,
on short settings.
"""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def check_common(d, steps, warmup):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["steps"] == steps and d["warmup"] == warmup and d["n_gpus"] == 1
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert "workload" in d["config"]
    e2e = d["e2e"]
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert key in e2e, key


def test_reference_arm_prints_the_contract_line():
    d = run_bench("--impl", "reference", "--workload", "single_head_f32", "--steps", "2", "--warmup", "1",
                  timeout=300)
    check_common(d, 2, 1)
    assert d["impl"] == "reference" and d["dtype"] == "f64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"]


@pytest.mark.gpu
def test_bench_line_carries_roofline_clocks_and_e2e():
    from tests.gpu_common import gpu_or_skip
    gpu_or_skip()
    d = run_bench("--steps", "20", "--warmup", "3", "--no-extra", "--no-cpu")
    check_common(d, 20, 3)
    assert d["dtype"] == "f16" and d["config"]["workload"] == "mha_f16_s4096"
    assert d["gpu_launches"] == 20
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert "traffic" in rf
    assert d["e2e"]["h2d_bytes_per_step"] == 3 * 16 * 4096 * 64 * 2
    assert d["e2e"]["d2h_bytes_per_step"] == 16 * 4096 * 64 * 2
    assert "clocks" in d


@pytest.mark.gpu
def test_bench_value_stays_above_the_committed_floor():
    """Performance regression check: the bench workload's throughput must stay
    within about 10 % of the last committed measurement (tests/perf_floor.json)."""
    from tests.gpu_common import gpu_or_skip
    gpu_or_skip()
    with open(os.path.join(ROOT, "tests", "perf_floor.json")) as f:
        floor = json.load(f)
    d = run_bench("--steps", "400", "--warmup", "5", "--no-extra", "--no-cpu")
    assert d["config"]["workload"] == floor["workload"]
    assert d["value"] >= floor["tflops_floor"], (d["value"], floor)
