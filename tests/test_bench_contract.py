"""The benchmark's output contract: one JSON line with the keys, types and units the
round's tooling reads.  The reference arm (the fp64 oracle on the host cores) runs on
the CPU; the native arm's line is checked on the GPU from a short run."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    return r


def _last_json(stdout):
    lines = [l for l in stdout.strip().splitlines() if l.startswith("{")]
    assert lines, stdout[-2000:]
    return json.loads(lines[-1])


def _check_common(d, steps, warmup):
    assert isinstance(d["metric"], str) and d["metric"]
    assert d["unit"] == "TFLOP/s"
    assert isinstance(d["value"], float) and d["value"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup
    assert d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["data"] == "synthetic" and isinstance(d["dtype"], str)
    assert isinstance(d["config"], dict) and d["config"]["workload"]
    e = d["e2e"]
    assert e["unit"] == d["unit"] and e["value"] > 0
    assert e["h2d_bytes_per_step"] >= 0 and e["d2h_bytes_per_step"] >= 0


def test_reference_arm_line():
    d = _last_json(_run(["--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-rows", "2"],
                        600).stdout)
    _check_common(d, 1, 3)
    assert d["impl"] == "reference" and d["dtype"] == "f64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"] and cb["sample"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_timing_rules_are_enforced():
    r = _run(["--impl", "reference", "--steps", "1", "--warmup", "0"], 300)
    assert r.returncode != 0 and "warmup" in r.stderr


@pytest.mark.gpu
def test_native_arm_line():
    r = _run(["--steps", "5", "--warmup", "3", "--no-rows", "--no-cpu-baseline"], 900)
    assert r.returncode == 0, r.stderr[-3000:]
    d = _last_json(r.stdout)
    _check_common(d, 5, 3)
    assert d.get("impl", "native") != "reference"
    rl = d["roofline"]
    assert rl["bound"] == "tensor" and rl["unit"] == "TFLOP/s" and rl["peak"] > 0
    assert abs(rl["frac"] - rl["achieved"] / rl["peak"]) < 1e-9
    assert 0.3 < rl["frac"] < 1.2
    assert rl["traffic"] is None or rl["traffic"] > 0
    assert d["gpu_launches"] >= d["steps"]
    c = d["clocks"]
    assert c["sm_max_mhz"] > 0 and isinstance(c["reasons"], list)
    e = d["e2e"]
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
