"""The bench's JSON-line contract on the CPU: the reference arm (the oracle timed
on host cores) prints one line with the required keys, and ranks other than 0
print nothing and exit 0."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None, *args):
    env = dict(os.environ)
    env.update(extra_env or {})
    env["MOE_REF_STEP_BUDGET_S"] = "0.05"
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", *args],
                       capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    return [ln for ln in p.stdout.splitlines() if ln.strip()]


def test_reference_arm_prints_one_contract_line():
    lines = _run()
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"].startswith("decode-40L")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    assert _run({"RANK": "1", "WORLD_SIZE": "2"}) == []


def test_cpu_baseline_samples_large_calls_and_times_small_ones_whole():
    sys.path.insert(0, ROOT)
    import bench
    import synth
    s = synth.Shape("cb", L=2, E=16, k=4, H=128, I=64, fmt=synth.FMT_MXFP4, act=synth.ACT_BF16, shared=1)
    whole = bench.cpu_baseline(s, 4, 2, budget_s=0.01)
    assert whole["kind"] == "oracle" and whole["value"] > 0 and "samples" not in whole["sample"]
    part = bench.cpu_baseline(s, 256, 2, budget_s=0.01)
    assert part["value"] > 0 and "samples" in part["sample"] and "1280" in part["sample"]
    assert bench.cpu_baseline(s, 4, 2, budget_s=0) is None
