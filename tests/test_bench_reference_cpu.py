"""bench.py's reference arm (the CPU oracle) on CPU: its JSON line and rank rule.

The reference arm times the oracle on the host cores on a bounded sample of
the workload and prints one JSON line with the same metric, unit and config
as the GPU arm; under a multi-rank launch only rank 0 prints.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as wl  # noqa: E402


def _run(extra_env=None, *args):
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    env.update(extra_env or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", *args], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    return [line for line in r.stdout.splitlines() if line.startswith("{")]


def test_reference_line_keeps_the_contract():
    lines = _run()
    assert len(lines) == 1
    d = json.loads(lines[0])
    w = wl.ALL_WORKLOADS[wl.BENCH_WORKLOAD]
    assert d["impl"] == "reference"
    assert d["metric"] == "fused B2B GEMM TFLOPS" and d["unit"] == "TFLOP/s"
    assert d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["steps"] == 1 and d["warmup"] >= 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"] == bench.workload_config(w, 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert cb["cores"] >= 1 and w.name in cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["vs_baseline"] is None


def test_reference_arm_prints_on_rank_zero_only():
    assert _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []


@pytest.mark.parametrize("name", ["tf32", "three_stage_bf16"])
def test_reference_arm_takes_any_workload(name):
    d = json.loads(_run(None, "--workload", name)[0])
    assert d["config"]["workload"] == name
    assert d["value"] > 0
