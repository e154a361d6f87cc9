"""bench.py's command-line contract on the CPU: the reference arm (the fp64
oracle timed on the host cores) prints one JSON line with the keys a
benchmark line carries, and the argument checks reject what the timing rules
forbid.  The GPU arm's line is checked where it runs (on a GPU)."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*argv, timeout=300):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *argv], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_one_complete_line():
    r = run_bench("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "unit", "config", "higher_is_better", "scaling", "dtype", "data"):
        assert k in d, k
    assert d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["ms_per_step"] > 0
    assert d["vs_baseline"] is None
    assert d["dtype"] == "f64"
    assert d["config"]["workload"] == "wan13_attn"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_too_few_warmup_steps_are_rejected():
    r = run_bench("--impl", "reference", "--steps", "1", "--warmup", "2", timeout=120)
    assert r.returncode == 2
    assert "--warmup must be >= 3" in r.stderr
