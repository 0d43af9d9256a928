"""The benchmark's output contract, checked on the CPU.

The reference arm (the oracle timed on the host cores) runs without a GPU,
so its JSON line, its rank handling and the warm-up rule can be checked here;
the algorithmic byte count the roofline uses is checked against its closed
form for the Llama-3-8B layer.
"""
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, env_extra=None, timeout=240):
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_one_contract_line():
    r = _bench("--impl", "reference", "--steps", "3", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["value"] > 0 and d["unit"] == "steps/s" and d["higher_is_better"] is True
    assert d["warmup"] == 3 and d["vs_baseline"] is None
    assert d["config"]["workload"] == "llama3-8b-layer-b8-ctx8k"
    # the GPU arm's config comes from the same function: the two lines agree
    import bench
    import workloads as W
    assert d["config"] == json.loads(json.dumps(bench.workload_config(W.WORKLOADS[1])))
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_fewer_than_three_warmup_steps_are_refused():
    r = _bench("--impl", "reference", "--steps", "3", "--warmup", "2")
    assert r.returncode != 0
    assert "warmup" in r.stderr


def test_reference_arm_runs_on_rank_zero_only():
    r = _bench("--impl", "reference", "--steps", "3", "--warmup", "3",
               env_extra={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [x for x in r.stdout.splitlines() if x.startswith("{")]


def test_step_bytes_closed_form_for_the_8b_layer():
    import bench
    import workloads as W
    w = W.WORKLOADS[1]
    # per unit: K and V of 1025 tokens, 12 B of metadata per token, q in and
    # out for 4 heads, the appended row written once
    per_unit = 2 * 1025 * 128 * 2 + 12 * 1025 + 2 * 4 * 128 * 2 + 2 * 128 * 2
    assert bench.step_bytes(w, np.full(64, 1025)) == 64 * per_unit == 34_538_240
