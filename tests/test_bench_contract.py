"""The benchmark's reference arm on the CPU: one JSON line with the keys the harness
reads (the GPU arm's line is produced on a GPU only)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["value"] > 0 and d["steps"] == 3 and d["warmup"] == 3
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_split_profiles_traffic_against_algorithmic_bytes():
    """The committed ncu summaries of the split pass: where one was taken on the current
    kernel source (the bench then reports its DRAM traffic), that traffic lies within 2 %
    above the launch's algorithmic bytes (every attended K and V row once, q, the lengths
    and the output). A summary taken on an older source is reported as a skip: the bench
    reports no traffic for it."""
    import pytest
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    stale = []
    for name in ("serving_mix", "llama3_8b_batched", "long_context_131k"):
        assert os.path.exists(bench.split_profile(name)), name
        traffic = bench.profiled_traffic(name)
        if traffic is None:
            stale.append(name)
            continue
        cfg = W.CONFIGS[name]
        lens = W.make_inputs(cfg, with_cache=False)["lens"].numpy()
        ratio = traffic / W.algorithmic_bytes(cfg, lens)["attn"]
        assert 1.0 <= ratio <= 1.02, (name, ratio)
    if stale:
        pytest.skip("summaries taken on another kernel source: " + ", ".join(stale))
