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
    assert cb["nproc"] >= 1 and "cpu_model" in cb
    # the steps it reports are the oracle layer calls it timed, in this run
    assert d["timed_s"] > 0 and d["ms_per_step"] * d["steps"] <= d["timed_s"] * 1e3 * 1.05 + 1
    assert d["config"]["pool_slots"] == 2560 and d["config"]["cache_flags"] == 0
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


def _fake_meas(T, K, L):
    R = K * L - 3  # calls whose experts all hit: the expert-kernel counters cover these
    timing = {"calls": K * L, "resident_calls": R, "route_ms": 0.02 * K * L, "gate_up_ms": 0.02 * R,
              "down_ms": 0.001 * R, "combine_ms": 0.0, "copy_ms": 0.3 * K,
              "gate_up_bytes": 10_000_000 * R, "down_bytes": 4_000_000 * R,
              "combine_bytes": 0, "copy_bytes": 13_000_000 * K}
    stats = {"hits": 300 * K, "misses": 8 * K, "prefetch_misses": 0, "bytes_h2d": 13_000_000 * K,
             "kernel_launches": 2 * K * L}
    return {"ms": 2.0 * K, "e2e_ms": 2.5 * K, "e2e_wall": 2.6 * K, "timing": timing, "stats": stats,
            "pcie": 52.0, "clk": {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "reasons": [], "samples": 5},
            "t_load": 12.0, "S": 2560, "frac": 0.25, "flags": 0, "L": L}


def test_bench_line_from_measurements():
    """The JSON line the GPU arm prints, built from fake counters on the CPU."""
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    K, L = 300, 40
    args = argparse.Namespace(workload="decode", steps=K, warmup=300, cpu_budget=0)
    d = bench.make_line(args, 1, _fake_meas(1, K, L), 1769984)
    json.dumps(d)
    assert d["value"] == round(K * 1 / (2.0 * K * 1e-3), 3) == 500.0
    assert d["ms_per_step"] == 2.0 and d["steps"] == K and d["warmup"] == 300
    assert d["e2e"]["value"] == 400.0 and d["e2e"]["h2d_bytes_per_step"] == L * 2048 * 2
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["kernel"].startswith("k_decode")
    assert r["algorithmic_bytes_per_launch"] == 14_000_000
    assert abs(r["achieved"] - 14_000_000 / 20e-6 / 1e9) < 0.1 and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-4
    assert d["gpu_launches"] == 2 * K * L and d["cpu_baseline"] is None
    assert d["cache"]["hit_rate"] == round(300 / 308, 4)
    assert "%d MB" % (308 * 1769984 // (1 << 20)) in d["config"]["l2"]
    # prefill: tensor roofline on the gate/up GEMM
    args = argparse.Namespace(workload="prefill", steps=3, warmup=3, cpu_budget=0)
    d = bench.make_line(args, 1, _fake_meas(4096, 3, 2), 6291456)
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and "tcgen05" in r["kernel"]
    assert r["algorithmic_flops_per_launch"] == 4.0 * 512 * 2048 * 4096 * 8


def test_dtype_strings_and_fp8_workloads():
    """The arithmetic each format's path computes in, as the JSON line states it,
    and the FP8 workloads registered with the stacks' shapes."""
    sys.path.insert(0, ROOT)
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    import synth
    assert bench._dtype_str(synth.FMT_BF16, 1) == "bf16 x bf16, fp32 accumulate"
    assert bench._dtype_str(synth.FMT_FP32, 4096) == "fp32"
    assert bench._dtype_str(synth.FMT_NVFP4, 1).startswith("nvfp4 weights") and "into f16" in bench._dtype_str(synth.FMT_NVFP4, 1)
    assert "fp8 weights (E4M3 code exact in f16" in bench._dtype_str(synth.FMT_FP8, 1)
    assert "exact in bf16" in bench._dtype_str(synth.FMT_FP8, 4096) and "bf16 activations" in bench._dtype_str(synth.FMT_FP8, 4096)
    assert "mxfp4" in bench._dtype_str(synth.FMT_MXFP4, 8)
    shape, T = bench.WORKLOADS["decode_fp8"][:2]
    assert shape.fmt == synth.FMT_FP8 and T == 1 and (shape.H, shape.E, shape.k, shape.I, shape.L) == (2048, 256, 8, 512, 40)
    shape, T = bench.WORKLOADS["prefill_fp8"][:2]
    assert shape.fmt == synth.FMT_FP8 and T == 4096
