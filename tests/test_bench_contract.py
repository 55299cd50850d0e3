"""The benchmark's reference arm (the oracle timed on the host cores) on the
smallest workload: one JSON line with the keys the benchmark contract names,
and no output from ranks other than 0 under a multi-process launch.  Runs on
the CPU (no GPU is touched by this arm)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["--impl", "reference", "--config", "tiny_f32", "--steps", "1", "--warmup", "3"]


def _bench(extra_env=None):
    env = dict(os.environ)
    env.update(extra_env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *ARGS], cwd=ROOT,
                          env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_json_line():
    r = _bench()
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["higher_is_better"] is True
    # steps and warmup are the oracle runs actually made (bounded by a time budget)
    assert d["n_gpus"] == 1 and d["steps"] >= 2 and d["warmup"] == 1 and d["extrapolated"]
    assert d["ms_per_step"] * d["steps"] <= d["wall_s"] * 1e3 * 1.01
    assert d["ms_per_step"] > 0 and d["vs_baseline"] is None and d["data"] == "synthetic"
    assert d["config"]["workload"].startswith("tiny_f32") and d["config"]["T"] == 256
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_print_nothing():
    r = _bench({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not r.stdout.strip()
