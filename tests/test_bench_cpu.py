"""The benchmark's contract on a machine without a GPU: the reference arm (the
CPU oracle) prints one JSON line with the keys the contract names, and the
library arm fails loudly instead of falling back to the CPU."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _run(*args, timeout=240):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_one_contract_line():
    r = _run("--impl", "reference", "--steps", "1", "--warmup", "1")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["steps"] == 1 and d["warmup"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == bench.WORKLOAD
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_library_arm_fails_without_gpu():
    r = _run("--steps", "1", "--warmup", "3", timeout=120)
    assert r.returncode != 0
    assert not any(ln.startswith("{") and '"value"' in ln for ln in r.stdout.splitlines())


def test_roofline_traffic_is_plausible():
    """The stored DRAM bytes per GEMM launch lie between the compulsory reads of
    the two operands and twice the algorithmic bytes of the step's shapes."""
    algo = [m * k + n * k + 2 * m * n for m, n, k in bench.shapes()]
    reads = [m * k + n * k for m, n, k in bench.shapes()]
    avg_algo = sum(algo) / len(algo)
    assert 0.5 * sum(reads) / len(reads) <= bench.GEMM_DRAM_BYTES_PER_LAUNCH <= 2 * avg_algo
