"""The bench's reference arm on the host (no GPU): `bench.py --impl
reference` times the fp64 oracle on a bounded sample of the workload and
prints one JSON line with the keys the bench contract names; a rank other
than 0 does no work and prints nothing."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(extra_env, *args):
    env = dict(os.environ, **extra_env)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                       capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    return [ln for ln in r.stdout.splitlines() if ln.strip()]


def test_reference_line():
    lines = run_bench({"RANK": "0"}, "--steps", "1", "--warmup", "1")
    d = json.loads(lines[-1])
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] >= 3  # the bench enforces three warm-up steps
    assert d["config"]["workload"].startswith("GRPO batch")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["ms_per_step"] > 0 and d["dtype"] == "f64" and d["data"] == "synthetic" and d["metric"]


def test_other_ranks_do_no_work():
    assert run_bench({"RANK": "1", "WORLD_SIZE": "2"}, "--steps", "1", "--warmup", "1") == []
