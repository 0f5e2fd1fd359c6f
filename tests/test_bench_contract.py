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


def test_accuracy_samples_report_exact_results_as_exact():
    """The bench's accuracy samples (evaluated in its CPU-baseline leg) give zero error
    when handed the oracle's own results, and see a planted error of the right size."""
    import numpy as np
    import torch

    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from context_exact_attention_gb300.workloads import make_qkv

    B, L, H, D = 1, 96, 3, 16
    q, k, v = make_qkv(B, L, H, D, seed=4, dtype=torch.bfloat16)
    rows = [0, 5, 95]
    ref, lref = oracle.attention(q, k, v, causal=True, rows=rows)
    got = torch.from_numpy(ref.copy())
    smp = bench.FwdSample(q, k, v, rows, got, torch.from_numpy(lref.copy()), True)
    acc = smp.evaluate(oracle)
    assert acc["max_abs"] == 0 and acc["lse_max_abs"] == 0 and abs(acc["cos"] - 1) < 1e-12
    bad = got.clone()
    bad[0, 1, 2, 3] += 0.25
    acc = bench.FwdSample(q, k, v, rows, bad, torch.from_numpy(lref.copy()), True).evaluate(oracle)
    assert abs(acc["max_abs"] - 0.25) < 1e-12 and acc["p3_ratio"] > 1
    both = bench.SegmentsSample([smp, smp]).evaluate(oracle)
    assert both["elements"] == 2 * got.numel() and both["max_abs"] == 0
    do = torch.randn(B, L, H, D, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    dref = oracle.attention_bwd_dq_rows(q, k, v, do, rows, causal=True)
    acc = bench.DqSample(q, k, v, do, rows, torch.from_numpy(dref.copy()), True).evaluate(oracle)
    assert acc["max_abs"] == 0
    oa, ob = torch.randn(7, D), torch.randn(7, D)
    la, lb = torch.randn(7), torch.randn(7)
    mo, ml = oracle.merge(oa, la, ob, lb)
    acc = bench.MergeSample(oa, la, ob, lb, torch.from_numpy(np.asarray(mo)),
                            torch.from_numpy(np.asarray(ml))).evaluate(oracle)
    assert acc["max_abs"] == 0 and acc["lse_max_abs"] == 0


@pytest.mark.gpu
def test_native_arm_line():
    r = _run(["--steps", "5", "--warmup", "3", "--no-rows", "--no-cpu-baseline",
              "--sustained-s", "0.5"], 900)
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
    assert c["samples"] >= c["samples_under_load"] >= 0
    su = d["sustained"]
    assert su["seconds"] >= 0.4 and su["value"] > 0 and su["unit"] == "TFLOP/s"
    assert abs(su["frac"] - su["value"] / su["peak"]) < 1e-9
    assert su["clocks"]["samples_under_load"] >= 1
    e = d["e2e"]
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
