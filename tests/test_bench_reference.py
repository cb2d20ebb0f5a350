"""bench.py's reference arm (the fp64 oracle timed on the host cores) runs
without a GPU: its one JSON line carries the keys of the benchmark contract,
and under a multi-rank launch only rank 0 prints."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None, *args):
    env = dict(os.environ)
    env.update(extra_env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--steps", "1", "--warmup", "3", *args],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_json_line():
    r = _run()
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference"
    for k in ("metric", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "dtype", "data", "config"):
        assert k in j, k
    assert j["value"] > 0 and j["ms_per_step"] > 0
    assert j["steps"] == 1 and j["warmup"] == 3 and j["n_gpus"] == 1
    assert j["vs_baseline"] is None
    assert j["config"]["workload"] == "serving_b128"
    # the same config object as the GPU arm's line (bench.config_of)
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_gqa_16_gb300 import workloads as wl
    assert j["config"] == bench.config_of(wl.make("serving_b128"), 1)
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == j["value"] and cb["unit"] == j["unit"]
    e = j["e2e"]
    assert e["value"] == j["value"] and e["unit"] == j["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_print_nothing():
    r = _run({"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"}, "--gpus", "2")
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]
