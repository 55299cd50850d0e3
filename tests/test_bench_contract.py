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


def _bench_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test",
                                                  os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_launch_count_matches_profiled_steps():
    """gpu_launches comes from launches_per_step(); its value for the two
    steps whose launch lists were profiled: 16 library kernels for a
    moe_s_bf16 step (one chunk, per-chunk weight gradients) and 132 for a
    long-context step (8 chunks of 32768 tokens, deferred weight gradients,
    stream-K router logits with their fix-up kernel on 152 SMs)."""
    b = _bench_module()
    from mixture_experts_layer_11_gb300 import synth
    assert b.launches_per_step(synth.CONFIGS["moe_s_bf16"], 1, False, False, False) == 16
    assert b.launches_per_step(synth.CONFIGS["longctx128_bf16"], 8, False, False, True) == 132
    # the permute fused into the GEMM loads removes one kernel per chunk
    assert b.launches_per_step(synth.CONFIGS["longctx128_bf16"], 8, False, False, True,
                               gather=True) == 124


def test_gemm_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    """roofline.traffic is read from the committed DRAM capture only while
    gemm_tc.cu is the source it was taken on (whitespace aside)."""
    import shutil
    b = _bench_module()
    from mixture_experts_layer_11_gb300 import synth
    cfg = synth.CONFIGS["longctx128_bf16"]
    n, note = b.gemm_traffic(cfg)
    assert n is not None and n > 0, note
    assert b.gemm_traffic(synth.CONFIGS["tiny_f32"])[0] is None   # no capture of it
    csrc = tmp_path / "mixture_experts_layer_11_gb300" / "csrc"
    csrc.mkdir(parents=True)
    shutil.copytree(os.path.join(ROOT, "profiles"), tmp_path / "profiles")
    src = open(os.path.join(ROOT, "mixture_experts_layer_11_gb300", "csrc", "gemm_tc.cu")).read()
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    (csrc / "gemm_tc.cu").write_text("\n\n  " + src.replace("\n", "\n ") + "\n")
    assert b.gemm_traffic(cfg)[0] == n                            # layout only
    (csrc / "gemm_tc.cu").write_text(src + "\n// changed\n")
    m, note = b.gemm_traffic(cfg)
    assert m is None and "changed" in note
