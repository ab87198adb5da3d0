"""The benchmark's reference arm on CPU: `bench.py --impl reference` times the
fp64 oracle on the host cores and prints the same one-line JSON contract as
the GPU arm; under a multi-rank launch only rank 0 works and prints."""
from __future__ import annotations

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3", "--reference-seconds", "1"]


def run_bench(args, env_extra=None):
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                          timeout=600, cwd=ROOT, env=env)


def json_lines(stdout):
    return [json.loads(line) for line in stdout.splitlines() if line.startswith("{")]


def test_reference_arm_prints_one_contract_line():
    r = run_bench(ARGS)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference"
    assert d["unit"] == "TFLOP/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["dtype"] == "f64" and d["vs_baseline"] is None
    assert d["config"]["B"] == 1 and d["config"]["N"] == 128 and d["config"]["D"] == 64
    base = d["cpu_baseline"]
    assert base["kind"] == "oracle" and base["cores"] >= 1 and base["value"] == d["value"] and base["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_without_work():
    r = run_bench(ARGS, {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert json_lines(r.stdout) == []
