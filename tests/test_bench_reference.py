"""The benchmark's reference arm (the fp64 CPU oracle, `bench.py --impl
reference`) on the CPU: it prints the contract's JSON line, and its per-step
sample is sized from a time budget, so that a large step count still ends in
bounded time."""
import json
import os
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, timeout=240):
    t0 = time.time()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                       capture_output=True, text=True, timeout=timeout, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    return line, time.time() - t0


@pytest.mark.parametrize("workload", ["stitch_64x30000", "bn_750000x32"])
def test_reference_line_and_bounded_time(workload):
    line, secs = _run("--workload", workload, "--steps", "400", "--warmup", "3", "--ref-budget", "3")
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["steps"] == 400 and line["warmup"] == 3
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    # 3 s of oracle time plus input generation and sizing; far below what
    # 403 whole-matrix steps would take
    assert secs < 120, secs


def test_reference_gemm_headline_defaults():
    line, secs = _run("--ref-budget", "4")
    assert line["unit"] == "TFLOP/s" and line["steps"] == 20 and line["warmup"] == 5
    assert line["config"]["M"] == 16384 and line["value"] > 0


def test_reference_under_two_ranks_prints_once():
    """Launched as two ranks (torchrun, CPU only): rank 0 alone runs the
    oracle and prints the line; the other rank exits 0 without work."""
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", "29531",
                        os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--workload", "stitch_64x30000", "--steps", "3", "--warmup", "3", "--ref-budget", "1"],
                       capture_output=True, text=True, timeout=240, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    assert json.loads(lines[0])["impl"] == "reference"


def test_ref_sample_size_fits_the_budget():
    """The sample-size search against a step whose cost is a + b n seconds
    (simulated by sleeping): the chosen n keeps calls x cost(n) within the
    budget, grows to n_max when the budget allows, and stays >= 1."""
    sys.path.insert(0, ROOT)
    import bench

    def make(a, b):
        def step_of(n):
            time.sleep(a + b * n)
        return step_of

    n = bench._ref_sample_size(make(0.0005, 0.0001), 10000, 40, 0.4)  # 10 ms a call: n <= 95
    assert 1 <= n <= 95 and 40 * (0.0005 + 0.0001 * n) <= 0.4 * 1.05
    assert bench._ref_sample_size(make(0.0, 1e-7), 64, 5, 10.0) == 64        # budget allows all
    assert bench._ref_sample_size(make(0.05, 0.0), 1000, 100, 0.1) == 1      # even one row is over
