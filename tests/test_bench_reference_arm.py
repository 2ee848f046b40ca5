"""bench.py --impl reference on the CPU: the oracle timed on a bounded
sample, printed as one JSON line with the keys of the libsp arm's line (same
metric, unit, direction and config object) plus its own cpu_baseline and e2e
blocks; under a multi-rank launch only rank 0 runs and prints."""
import json
import os
import subprocess
import sys

from conftest import ROOT

REQUIRED = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config")


def run_bench(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--config", "tiny", *args], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=600)


def test_reference_arm_line():
    r = run_bench({}, "--steps", "2", "--warmup", "1")
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in REQUIRED:
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    assert d["unit"] == "branch tokens/s" and d["higher_is_better"] is True
    assert d["value"] > 0
    assert d["config"]["workload"].startswith("tiny: Hq 8/Hkv 2/d 64, 4 branches")
    assert d["config"]["branch_tokens_per_step"] == 128
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_do_nothing():
    r = run_bench({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--steps", "1",
                  "--warmup", "0", "--gpus", "2")
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
