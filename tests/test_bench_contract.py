"""The benchmark's reference arm on CPU (the fp64 oracle on bounded samples of
the headline workload): one JSON line with the keys and units the GPU arm
also prints, so both arms can be compared by the same reader."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["unit"] == "µs/call" and d["higher_is_better"] is False
    assert d["steps"] == 1 and d["warmup"] == 3 and d["value"] > 0
    assert abs(d["ms_per_step"] * 1e3 - d["value"]) <= 1e-3 * d["value"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["sample"]
    # timed on every host core the process may use, the 1-core time beside it
    assert cb["cores"] == len(os.sched_getaffinity(0))
    assert cb["single_core"]["cores"] == 1 and cb["single_core"]["value"] > 0
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert "workload" in d["config"]


def test_bench_refuses_fewer_than_three_warmup_steps():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "2"], cwd=ROOT, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode != 0 and "warmup" in r.stderr
