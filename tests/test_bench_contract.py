"""bench.py's output contract, checked on the host.

The reference arm (the oracle timed on the host cores) prints one JSON line
with every key of the contract, its cpu_baseline and e2e describing the same
run; under several ranks only rank 0 prints; and the native arm on a machine
without a GPU stops with an error instead of falling back to the CPU."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches")


def _bench(args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, "bench.py"] + args, cwd=ROOT, capture_output=True, text=True,
                          timeout=600, env=e)


def _json_lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def test_reference_arm_prints_one_complete_line():
    r = _bench(["--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert all(k in d for k in KEYS), [k for k in KEYS if k not in d]
    assert d["impl"] == "reference"
    assert (d["steps"], d["warmup"], d["n_gpus"]) == (2, 3, 1)
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["dtype"] == "f64" and d["gpu_launches"] == 0 and d["vs_baseline"] is None
    assert d["config"]["workload"] and "model" not in d["config"]
    # one token per step on this workload: value x seconds per step = 1
    assert d["value"] * d["ms_per_step"] * 1e-3 == pytest.approx(1.0, rel=1e-9)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e2e = d["e2e"]
    assert (e2e["value"], e2e["unit"]) == (d["value"], d["unit"])
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_print_nothing():
    r = _bench(["--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "3"],
               env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour on a machine without a GPU")
def test_native_arm_without_a_gpu_fails_loudly():
    r = _bench(["--steps", "1", "--warmup", "3", "--no-cpu"])
    assert r.returncode != 0
    assert _json_lines(r.stdout) == []
