"""bench.py's JSON line on the CPU: the reference arm (the oracle) on the
router-only workload prints one line with the keys the benchmark contract
fixes, and the workload table names every configuration the generator has."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_reference_arm_line_keys():
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "k2_router", "--steps", "2", "--warmup", "1"],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["name"] == "k2_router" and "workload" in d["config"]


def test_workloads_cover_the_generator_configs():
    gpu_configs = set(synth.CONFIGS) - {"tiny"}  # tiny: a parity case, not a bench line
    assert gpu_configs <= set(bench.WORKLOADS)


def test_per_step_work_counts_fp8_weight_bytes():
    import numpy as np
    bf = synth.shape("k2_decode")
    f8 = synth.shape("k2_decode_fp8")
    counts = np.zeros(bf.E_routed, dtype=np.int64)
    counts[:10] = 5
    wb = bench.per_step_work(bf, counts)
    w8 = bench.per_step_work(f8, counts)
    # same flops; FP8 weights are one byte per weight plus a 4-byte scale per 128 x 128 block
    assert w8["flops_layer"] == wb["flops_layer"]
    per_expert_bf16 = 3 * bf.d_ff * bf.d_model * 2
    per_expert_fp8 = 3 * bf.d_ff * bf.d_model * (1 + 4 / (128 * 128))
    want = wb["layer_bytes"] - 11 * (per_expert_bf16 - per_expert_fp8)  # 10 routed + 1 shared
    assert abs(w8["layer_bytes"] - want) <= 2
