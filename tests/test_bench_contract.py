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


def test_frame_and_slot_accounting_pins():
    """The conversions the DiT legs report, pinned to the pages' numbers
    ("Wave Forcing"): 399 latent frames are saved as 1593 video frames
    (App. C, VBench-Long protocol: 133 chunks of 3 latent frames, 1 + 398 x 4),
    so a steady chunk adds 12 video frames; a 133-chunk request at S = 4
    keeps 133 / 137 = 97.1% of its stage slots busy (App. B.4 Eq. 16); and
    Table 4 (App. C.2) reports steady FPS as 12 frames per tick: tick p50
    78.88 ms -> 152.13 FPS, 76.05 ms -> 157.79, 120.53 ms -> 99.56."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.video_frames(133, 3) == 1593
    assert bench.video_frames(134, 3) - bench.video_frames(133, 3) == 12
    assert bench.frames_per_s(1.0, 3) == 12
    assert bench.frames_per_s(6.0, 3) == 72
    assert round(100 * bench.eta_slot(133, 4), 1) == 97.1
    assert bench.eta_slot(133, 4) == 133 / 137
    assert bench.eta_slot(10, 4, sequential=True) == 1 / 5
    for tick_ms, fps in ((78.88, 152.13), (76.05, 157.79), (120.53, 99.56)):
        assert round(bench.frames_per_s(1000.0 / tick_ms), 2) == fps, tick_ms
    # the rate a chunk rate implies agrees with the frame count a request implies
    n, seconds = 133, 20.0
    assert abs(bench.frames_per_s(n / seconds) * seconds - (bench.video_frames(n) + 3)) < 1e-9
