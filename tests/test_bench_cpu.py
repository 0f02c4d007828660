"""bench.py on a machine without a GPU.

The reference arm (the fp64 oracle on the host cores, on sampled rows of the
benchmark's workload) prints its one JSON line with the keys the benchmark
contract names; the library arm fails with an error instead of falling back to
a CPU computation.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="checks the behaviour without a GPU")


def run_bench(args, timeout):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=timeout)


def json_lines(text):
    return [line for line in text.splitlines() if line.startswith("{")]


def test_reference_arm_prints_its_line():
    r = run_bench(["--impl", "reference", "--steps", "1", "--warmup", "0"], 900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = json_lines(r.stdout)
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 0
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "attn_bf16_causal_b2h32n4096d128"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_library_arm_fails_without_gpu():
    r = run_bench(["--steps", "1", "--warmup", "0"], 300)
    assert r.returncode != 0
    assert not json_lines(r.stdout)
