"""Benchmark: exact ring-attention forward on GB300, one JSON line on stdout.

Headline workload: causal LM context-parallel forward, B=1, H=32, L=32768, D=128,
bf16, P=8 virtual ring shards of 4096 tokens with whole-shard causal skip
(q, k ~ N(0,1) scaled per head by s_h ~ U[0.5, 2], v ~ N(0,1)).  One step is
one ring_attn_fwd call over that input; the metric is algorithmic TFLOP/s
(4*D per visible query/key pair).  Inputs (3 x 256 MiB) exceed the 129 MB L2,
so no flush is needed between steps.

Also measured in the same run (the "rows" object): the diffusion-DiT full
attention workload (40 calls), the LSE merge at the causal-LM size, the Ulysses
transposes and pipeline, the backward of the causal-LM workload, and the
long-context causal workload.

--impl reference times the fp64 CPU oracle (the only reference this project
has) on the host cores, on a bounded sample of query rows of the same workload.
Multi-GPU (torchrun): every rank runs the same workload on its own GPU
(independent replicas, weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from context_exact_attention_gb300.workloads import (DIT, LM, LONG, ULYSSES,  # noqa: E402
                                                     attention_flops, make_workload_inputs,
                                                     sample_rows)

METRIC = "attention fwd TFLOP/s (bf16, full & causal) and % of GB300 dense BF16 peak"
HEADLINE = LM
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SRC = os.path.join(ROOT, "context_exact_attention_gb300", "csrc", "attn_bf16_sm103.cu")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
E2E_HEADS_PER_GROUP = 4   # head-group size of the host-buffer entry point in the e2e leg


def _rank_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def _peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def _kernel_hash():
    with open(KERNEL_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def _forward_kernel_name(w):
    """The forward kernel a contiguous bf16 call of workload w runs: head dim 128 with
    key walks of 8192 keys or more go to the pair-of-SMs kernel."""
    if w.D == 128 and w.L >= 8192:
        return "ring_attn_bf16_pair_kernel<0>"
    return f"ring_attn_bf16_kernel<{w.D}, 0>"


def _traffic_per_launch():
    """DRAM bytes of one ring_attn_fwd launch from a committed ncu summary, if it was
    taken on the current kernel source; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        if t.get("kernel_sha256_16") == _kernel_hash():
            return t.get("bytes_per_launch_full_workload")
    except (OSError, ValueError):
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clock, utilisation, power and throttle reasons while a
    timed loop runs (every 50 ms).  The summary's sm_mhz is the median over the samples
    taken under load (GPU utilisation >= 50 %), so idle samples before and after the
    loop do not enter it; reasons are those seen in any sample."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def __enter__(self):
        exe = shutil.which("nvidia-smi")
        if exe:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen([exe, f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                                          "-lms", "50"], stdout=self.out,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    @staticmethod
    def _num(x):
        return float(x.split()[0])

    def summary(self):
        if not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 11:
                    continue
                if self.uuid and parts[1] != self.uuid:
                    continue
                try:
                    rows.append({"sm": self._num(parts[2]), "max": self._num(parts[3]),
                                 "power": self._num(parts[4]), "util": self._num(parts[5]),
                                 "reasons": [n for n, v in zip(self.REASONS, parts[7:11])
                                             if v.lower() == "active"]})
                except (ValueError, IndexError):
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r["util"] >= 50]
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded) if loaded else None,
                "sm_mhz_min_under_load": min(r["sm"] for r in loaded) if loaded else None,
                "sm_max_mhz": max(r["max"] for r in rows),
                "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(r["power"] for r in rows),
                "reasons": sorted({n for r in rows for n in r["reasons"]}),
                "reasons_under_load": sorted({n for r in loaded for n in r["reasons"]})}


def _time_loop(fn, steps, stream):
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn()
    stop.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(stop)


def max_over_ranks(ms, dist=None):
    """The slowest rank's time (the whole job ends when its last rank does)."""
    if dist is None:
        return ms
    t = torch.tensor([ms], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _flops_rows(L, D, causal, rows, heads):
    per_head = sum((i + 1) if causal else L for i in rows)
    return 4 * D * heads * per_head


def cpu_oracle_sample(w, budget_s=15.0, seed=0):
    """Time the fp64 oracle on the host cores on sampled query rows of workload w.
    Returns (TFLOP/s, seconds, rows, threads)."""
    import oracle

    q, k, v = (oracle.to_f64(t) for t in make_workload_inputs(w, seed=seed))
    threads = oracle.default_threads()
    probe = sample_rows(w.L, w.P, 2 * w.P, seed=1)        # shard edges only
    t0 = time.perf_counter()
    oracle.attention(q, k, v, causal=w.causal, rows=probe, threads=threads)
    dt = max(time.perf_counter() - t0, 1e-3)
    per_row = dt / len(probe)
    n = int(max(2 * w.P, min(4 * w.L, budget_s / per_row)))
    rows = sample_rows(w.L, w.P, n, seed=1)
    t0 = time.perf_counter()
    oracle.attention(q, k, v, causal=w.causal, rows=rows, threads=threads)
    dt = time.perf_counter() - t0
    fl = _flops_rows(w.L, w.D, w.causal, rows, w.B * w.H)
    return fl / dt / 1e12, dt, len(rows), threads


class FwdSample:
    """Host copies of what the oracle needs to check a few query rows of one forward
    result: q, k, v of the chosen heads (position order), the query rows (positions),
    and the GPU's out / lse at those rows.  Evaluated only in the CPU-baseline leg."""

    def __init__(self, q, k, v, rows, out_rows, lse_rows, causal):
        self.q, self.k, self.v = q, k, v
        self.rows, self.out, self.lse, self.causal = list(rows), out_rows, lse_rows, causal

    def evaluate(self, oracle):
        ref, lref = oracle.attention(self.q, self.k, self.v, causal=self.causal, rows=self.rows)
        return _accuracy(self.out, ref, self.lse, lref)


class SegmentsSample:
    """A packed-sequence result: one FwdSample per sequence (that sequence alone)."""

    def __init__(self, parts):
        self.parts = parts

    def evaluate(self, oracle):
        acc = [p.evaluate(oracle) for p in self.parts]
        return _combine_accuracy(acc)


class DqSample:
    """dq of a few query rows of a backward result (chosen heads), against the oracle's
    per-row chain rule."""

    def __init__(self, q, k, v, do, rows, dq_rows, causal):
        self.q, self.k, self.v, self.do = q, k, v, do
        self.rows, self.dq, self.causal = list(rows), dq_rows, causal

    def evaluate(self, oracle):
        ref = oracle.attention_bwd_dq_rows(self.q, self.k, self.v, self.do, self.rows,
                                           causal=self.causal)
        return _accuracy(self.dq, ref)


class MergeSample:
    """A few rows of an LSE merge and its inputs."""

    def __init__(self, oa, la, ob, lb, oo, lo):
        self.args, self.oo, self.lo = (oa, la, ob, lb), oo, lo

    def evaluate(self, oracle):
        ref, lref = oracle.merge(*self.args)
        return _accuracy(self.oo, ref, self.lo, lref)


def _accuracy(got, ref, got_lse=None, ref_lse=None):
    import numpy as np

    g = got.double().numpy() if hasattr(got, "double") else np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64).reshape(g.shape)
    err = np.abs(g - r)
    res = {"elements": int(g.size), "max_abs": float(err.max()),
           "p3_ratio": float((err / (5e-3 + 5e-3 * np.abs(r))).max()),
           "cos": float((g * r).sum() / np.sqrt((g * g).sum() * (r * r).sum()))}
    if got_lse is not None:
        gl = got_lse.double().numpy()
        res["lse_max_abs"] = float(np.abs(gl - np.asarray(ref_lse, np.float64).reshape(gl.shape)).max())
    return res


def _combine_accuracy(parts):
    res = {"elements": sum(p["elements"] for p in parts),
           "max_abs": max(p["max_abs"] for p in parts),
           "p3_ratio": max(p["p3_ratio"] for p in parts),
           "cos": min(p["cos"] for p in parts)}
    if all("lse_max_abs" in p for p in parts):
        res["lse_max_abs"] = max(p["lse_max_abs"] for p in parts)
    return res


def _host(t):
    return t.detach().to("cpu", copy=True)


def _fwd_sample(q, k, v, out, lse, rows, heads, causal, kv_heads=None):
    """FwdSample of query rows `rows` (position order) of heads `heads` of a [B, L, H, D]
    result; kv_heads: the key/value heads those query heads read (default: the same)."""
    kv_heads = heads if kv_heads is None else kv_heads
    idx = torch.tensor(rows, device=out.device)
    return FwdSample(_host(q[:, :, heads]), _host(k[:, :, kv_heads]), _host(v[:, :, kv_heads]),
                     rows, _host(out[:, idx][:, :, heads]), _host(lse[:, idx][:, :, heads]),
                     causal)


def run_reference(args, rank, world):
    """fp64 CPU oracle arm: each step is a bounded sample of query rows of the workload."""
    if rank != 0:
        return
    import oracle

    w = HEADLINE
    q, k, v = (oracle.to_f64(t) for t in make_workload_inputs(w, seed=0))
    threads = oracle.default_threads()
    n_rows = args.ref_rows
    rows_all = sample_rows(w.L, w.P, n_rows * (args.warmup + args.steps), seed=1)
    chunks = [rows_all[i::args.warmup + args.steps] for i in range(args.warmup + args.steps)]
    for c in chunks[:args.warmup]:
        oracle.attention(q, k, v, causal=w.causal, rows=c, threads=threads)
    fl = 0
    t0 = time.perf_counter()
    for c in chunks[args.warmup:]:
        oracle.attention(q, k, v, causal=w.causal, rows=c, threads=threads)
        fl += _flops_rows(w.L, w.D, w.causal, c, w.B * w.H)
    dt = time.perf_counter() - t0
    value = fl / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "L": w.L, "H": w.H, "D": w.D, "P": w.P,
                   "causal": w.causal, "sample": f"{n_rows} query rows x {w.B * w.H} heads per step"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n_rows} sampled query rows (all heads) per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_gpu(args, rank, world, local_rank):
    import context_exact_attention_gb300 as cea

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cea.load_library()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")

    w = HEADLINE
    if args.profile_case:
        w = dataclasses.replace(w, H=8, name=w.name.replace("H32", "H8") + " (profile case)")
    qc, kc, vc = make_workload_inputs(w, seed=0)
    q, k, v = (t.to(dev) for t in (qc, kc, vc))
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.L, w.H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    step = lambda: cea.ring_attn_fwd(q, k, v, P=w.P, causal=w.causal, out=out, lse=lse,
                                      stream=stream)
    for _ in range(args.warmup):
        step()
    if cea.check_status(stream) != 0:
        raise RuntimeError("kernel reported a device-side timeout during warm-up")
    flops = attention_flops(w.B, w.L, w.H, w.D, w.causal)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    if dist is not None:
        dist.barrier()
    with ClockSampler(uuid) as clk:
        ms = _time_loop(step, args.steps, stream)
    clocks = clk.summary()
    if cea.check_status(stream) != 0:
        raise RuntimeError("kernel reported a device-side timeout in the timed region")
    ms_max = max_over_ranks(ms, dist)
    ms_step = ms_max / args.steps
    value = flops * world / (ms_step * 1e-3) / 1e12

    # the same step back to back for >= sustained_s seconds: the figure at the power cap
    # (the short headline loop is a burst figure), with its own clock record
    sustained = None
    if args.sustained_s > 0:
        n_sus = max(args.steps, int(args.sustained_s * 1e3 / ms_step) + 1)
        with ClockSampler(uuid) as clk2:
            ms_sus = _time_loop(step, n_sus, stream) / n_sus
        sustained = {"steps": n_sus, "ms_per_step": ms_sus, "seconds": ms_sus * n_sus / 1e3,
                     "value": flops / (ms_sus * 1e-3) / 1e12, "clocks": clk2.summary()}
        if cea.check_status(stream) != 0:
            raise RuntimeError("kernel reported a device-side timeout in the sustained loop")

    # host copy of the result on sampled rows, checked against the oracle in the
    # CPU-baseline leg (inputs qc, kc, vc are already on the host)
    acc_rows = sample_rows(w.L, w.P, args.acc_rows, seed=1)
    ridx = torch.tensor(acc_rows, device=dev)
    samples = {"headline": FwdSample(qc, kc, vc, acc_rows, _host(out[:, ridx]), _host(lse[:, ridx]),
                                     w.causal)}

    # -- end to end through the public API: pinned host inputs in, host results out.
    # ring_attn_fwd_host copies head groups in, runs the attention and copies the results
    # back inside the call, overlapping the three; the device workspace is allocated once.
    hq, hk, hv = (t.pin_memory() for t in (qc, kc, vc))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    group = E2E_HEADS_PER_GROUP if w.H % E2E_HEADS_PER_GROUP == 0 else 1
    ws = torch.empty(cea.host_workspace_bytes(w.B, w.L, w.H, w.D, group), dtype=torch.uint8,
                     device=dev)
    del q, k, v, out, lse   # the device copies of the timed step are not needed any more

    def e2e_step():
        cea.ring_attn_fwd_host(hq, hk, hv, P=w.P, causal=w.causal, out=hout, lse=hlse,
                               heads_per_group=group, workspace=ws, stream=stream)

    for _ in range(2):
        e2e_step()
    e2e_steps = max(3, args.steps // 4)
    # one event between consecutive steps (same stream, no synchronisation): the loop's
    # total gives the metric; the per-step times give the median and the slowest step
    # beside it, since the CPU-GPU link can stall for tens of milliseconds now and then
    e2e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps + 1)]
    torch.cuda.synchronize()
    e2e_ev[0].record(stream)
    for i in range(e2e_steps):
        e2e_step()
        e2e_ev[i + 1].record(stream)
    torch.cuda.synchronize()
    e2e_each = [e2e_ev[i].elapsed_time(e2e_ev[i + 1]) for i in range(e2e_steps)]
    e2e_ms = e2e_ev[0].elapsed_time(e2e_ev[-1]) / e2e_steps
    e2e_median = sorted(e2e_each)[e2e_steps // 2]
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = hout.numel() * hout.element_size() + hlse.numel() * hlse.element_size()

    peaks, peak_src = _peaks()
    peak = float(peaks["bf16_tflops"])
    peak_sus = float(peaks.get("bf16_tflops_sustained", peak))
    achieved = flops / (ms_step * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": _traffic_per_launch(),
                "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json)" if peak_src == "measured"
                else "fallback 1.9 PFLOP/s bf16",
                "frac_of_sustained": achieved / peak_sus,
                "kernel": _forward_kernel_name(w)}
    if sustained is not None:
        sustained.update({"unit": "TFLOP/s", "peak": peak_sus,
                          "frac": sustained["value"] / peak_sus,
                          "frac_of_burst": sustained["value"] / peak,
                          "peak_source": f"{peak_src} bf16 sustained (MEASURED_PEAKS.json)"})

    rows = {}
    if not args.no_rows and rank == 0:
        rows = measure_rows(cea, dev, stream, peaks, samples)

    cpu = None
    accuracy = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, dt, n, threads = cpu_oracle_sample(w, budget_s=args.cpu_budget)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{n} sampled query rows x {w.B * w.H} heads of the causal-LM workload "
                         f"({dt:.1f} s, fp64)"}
        # the GPU results on sampled rows against the fp64 oracle (not timed)
        import oracle

        for name, smp in samples.items():
            acc = smp.evaluate(oracle)
            if name == "headline":
                accuracy = dict(acc, rows=len(acc_rows), heads=w.H,
                                tolerance="|err| <= 5e-3 + 5e-3 |ref| (p3_ratio <= 1), cos > 0.999")
            elif name in rows:
                rows[name]["accuracy"] = acc

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "L": w.L, "H": w.H, "D": w.D, "P": w.P,
                       "causal": w.causal, "global_batch": w.B * world, "seq_len": w.L,
                       "parallelism": f"replicas{world}",
                       "l2": f"inputs {3 * hq.numel() * 2 / 1e6:.0f} MB per step > 129 MB L2 "
                             "(no flush needed)"},
            "roofline": roofline, "sustained": sustained, "cpu_baseline": cpu,
            "accuracy": accuracy,
            "e2e": {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms, "median_ms_per_step": e2e_median,
                    "max_ms_per_step": max(e2e_each),
                    "api": f"ring_attn_fwd_host, pinned host buffers, heads_per_group={group}"},
            "gpu_launches": args.steps, "clocks": clocks, "rows": rows,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def measure_rows(cea, dev, stream, peaks, samples):
    """Secondary measurements: every other hot-path row, a few timed repetitions each.
    Each row also leaves in `samples` a host copy of its result on a few sampled rows, for
    the accuracy check of the CPU-baseline leg."""
    res = {}
    hbm = float(peaks["hbm_gbs"])
    peak = float(peaks["bf16_tflops"])

    # diffusion-DiT full attention, 40 calls as one denoising loop
    w = DIT
    q, k, v = (t.to(dev) for t in make_workload_inputs(w, seed=0))
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.L, w.H), dtype=torch.float32, device=dev)
    f = lambda: cea.ring_attn_fwd(q, k, v, P=w.P, causal=False, out=out, lse=lse, stream=stream)
    for _ in range(3):
        f()
    ms = _time_loop(f, w.repeats, stream)
    fl = attention_flops(w.B, w.L, w.H, w.D, False)
    res["dit_full_x40"] = {"ms_total": ms, "ms_per_call": ms / w.repeats,
                           "tflops": fl * w.repeats / (ms * 1e-3) / 1e12,
                           "frac": fl * w.repeats / (ms * 1e-3) / 1e12 / peak,
                           "note": "inputs 72 MiB fit in L2; back-to-back calls"}
    samples["dit_full_x40"] = _fwd_sample(q, k, v, out, lse, sample_rows(w.L, w.P, 16, seed=1),
                                          [0, 13], False)
    del q, k, v, out, lse

    # LSE merge at the causal-LM size: two partials of 1,048,576 rows x 128 bf16
    rows, D = LM.B * LM.L * LM.H, LM.D
    g = torch.Generator(device=dev).manual_seed(0)
    oa = torch.randn(rows, D, device=dev, generator=g).to(torch.bfloat16)
    ob = torch.randn(rows, D, device=dev, generator=g).to(torch.bfloat16)
    la = torch.randn(rows, device=dev, generator=g)
    lb = torch.randn(rows, device=dev, generator=g)
    oo, lo = torch.empty_like(oa), torch.empty_like(la)
    f = lambda: cea.attn_merge_partials(oa, la, ob, lb, o_out=oo, lse_out=lo, stream=stream)
    for _ in range(3):
        f()
    n = 20
    ms = _time_loop(f, n, stream) / n
    by = rows * (3 * D * 2 + 3 * 4)
    res["merge_lm_size"] = {"ms": ms, "GB/s": by / (ms * 1e-3) / 1e9,
                            "frac": by / (ms * 1e-3) / 1e9 / hbm, "bytes": by,
                            "note": "working set 805 MB > L2"}
    pick = torch.randperm(rows, generator=torch.Generator().manual_seed(3))[:64].to(dev)
    samples["merge_lm_size"] = MergeSample(*(_host(t[pick]) for t in (oa, la, ob, lb, oo, lo)))
    del oa, ob, la, lb, oo, lo

    # Ulysses transposes and pipeline
    w = ULYSSES
    Ls, Hg = w.L // w.P, w.H // w.P
    x = torch.randn(w.P, w.B, Ls, w.H, w.D, device=dev, generator=g).to(torch.bfloat16)
    y = torch.empty(w.P, w.B, w.L, Hg, w.D, device=dev, dtype=torch.bfloat16)
    f = lambda: cea.ulysses_seq2head(x, w.P, out=y, stream=stream)
    for _ in range(3):
        f()
    ms = _time_loop(f, n, stream) / n
    by = 2 * x.numel() * 2
    res["ulysses_seq2head"] = {"ms": ms, "GB/s": by / (ms * 1e-3) / 1e9,
                               "frac": by / (ms * 1e-3) / 1e9 / hbm, "bytes": by}
    f = lambda: cea.ulysses_head2seq(y, w.P, out=x, stream=stream)
    ms = _time_loop(f, n, stream) / n
    res["ulysses_head2seq"] = {"ms": ms, "GB/s": by / (ms * 1e-3) / 1e9,
                               "frac": by / (ms * 1e-3) / 1e9 / hbm, "bytes": by}
    qs = x
    ks = torch.randn_like(x, dtype=torch.float32).to(torch.bfloat16)
    vs = torch.randn_like(x, dtype=torch.float32).to(torch.bfloat16)
    bufs = {nm: torch.empty(w.P, w.B, w.L, Hg, w.D, device=dev, dtype=torch.bfloat16)
            for nm in ("q", "k", "v", "o")}
    f = lambda: cea.ulysses_attention(qs, ks, vs, w.P, stream=stream, buffers=bufs)
    for _ in range(2):
        f()
    n2 = 5
    ms = _time_loop(f, n2, stream) / n2
    fl = attention_flops(w.B, w.L, w.H, w.D, False)
    res["ulysses_pipeline"] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                               "frac": fl / (ms * 1e-3) / 1e12 / peak,
                               "note": "3 seq2head + attention (B'=16, H'=4, P=1) + head2seq"}
    # the same step in one kernel: the transposes folded into the tensor maps' addressing
    o_seq = torch.empty_like(qs)
    f = lambda: cea.ulysses_attention_fused(qs, ks, vs, w.P, out=o_seq, stream=stream)
    for _ in range(2):
        f()
    ms = _time_loop(f, n2, stream) / n2
    res["ulysses_fused"] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                            "frac": fl / (ms * 1e-3) / 1e12 / peak,
                            "note": "ulysses_attention_fused: same result, no head-sharded copies"}
    # position order [B, L, H, D]: position r * L/P + i of batch b is row i of shard r
    seq_to_pos = lambda t: t.permute(1, 0, *range(2, t.dim())).reshape(w.B, w.L, *t.shape[3:])
    _, lse_seq = cea.ulysses_attention_fused(qs, ks, vs, w.P, out=o_seq, want_lse=True,
                                             stream=stream)
    samples["ulysses_fused"] = _fwd_sample(seq_to_pos(qs), seq_to_pos(ks), seq_to_pos(vs),
                                           seq_to_pos(o_seq), seq_to_pos(lse_seq),
                                           sample_rows(w.L, w.P, 16, seed=1), [0, 21], False)
    del x, y, qs, ks, vs, bufs, o_seq

    # grouped key/value heads at the headline shape: 32 query heads over 8 key/value heads
    w = LM
    q, _, _ = (t.to(dev) for t in make_workload_inputs(w, seed=0))
    kk = torch.randn(w.B, w.L, 8, w.D, device=dev, generator=g).to(torch.bfloat16)
    vv = torch.randn(w.B, w.L, 8, w.D, device=dev, generator=g).to(torch.bfloat16)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.L, w.H), dtype=torch.float32, device=dev)
    f = lambda: cea.ring_attn_fwd_gqa(q, kk, vv, P=w.P, causal=True, out=out, lse=lse,
                                      stream=stream)
    f()
    ms = _time_loop(f, 5, stream) / 5
    fl = attention_flops(w.B, w.L, w.H, w.D, True)
    res["lm_gqa_32q_8kv"] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                             "frac": fl / (ms * 1e-3) / 1e12 / peak}
    samples["lm_gqa_32q_8kv"] = _fwd_sample(q, kk, vv, out, lse, sample_rows(w.L, w.P, 16, seed=1),
                                            [0, 21], True, kv_heads=[0, 5])
    del q, kk, vv, out, lse

    # zigzag layout of the headline workload (shard r holds chunks r and 2P-1-r)
    w = LM
    q, k, v = (t.to(dev) for t in make_workload_inputs(w, seed=0))
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.L, w.H), dtype=torch.float32, device=dev)
    f = lambda: cea.ring_attn_fwd_zigzag(q, k, v, P=w.P, out=out, lse=lse, stream=stream)
    f()
    ms = _time_loop(f, 5, stream) / 5
    fl = attention_flops(w.B, w.L, w.H, w.D, True)
    res["lm_zigzag"] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                        "frac": fl / (ms * 1e-3) / 1e12 / peak}
    # zigzag row i holds position pos[i]: position order is the inverse permutation
    inv = torch.argsort(torch.tensor(cea.zigzag_positions(w.L, w.P))).to(dev)
    samples["lm_zigzag"] = _fwd_sample(q[:, inv], k[:, inv], v[:, inv], out[:, inv], lse[:, inv],
                                       sample_rows(w.L, w.P, 16, seed=1), [2, 30], True)
    del q, k, v, out, lse

    # packed variable-length sequences filling the headline length (causal)
    w = LM
    lengths, cu = packed_lengths(w.L)
    cu_d = torch.tensor(cu, dtype=torch.int32, device=dev)
    q, k, v = (torch.randn(w.L, w.H, w.D, device=dev, generator=g).to(torch.bfloat16)
               for _ in range(3))
    out = torch.empty_like(q)
    lse = torch.empty((w.L, w.H), dtype=torch.float32, device=dev)

    def f():
        # the heaviest-first unit order is computed from cu_seqlens inside every step
        sched = cea.varlen_schedule(cu_d, w.L, w.P, True, stream=stream)
        cea.ring_attn_fwd_varlen(q, k, v, cu_d, P=w.P, causal=True, out=out, lse=lse,
                                 stream=stream, schedule=sched)
    f()
    ms = _time_loop(f, 5, stream) / 5
    fl = sum(attention_flops(1, n, w.H, w.D, True) for n in lengths)
    res["lm_varlen_causal"] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                               "frac": fl / (ms * 1e-3) / 1e12 / peak, "n_seqs": len(lengths),
                               "note": "lengths U[256, 8192) packed to 32768 tokens, 32 heads; "
                                       "schedule computed in each step"}
    picked = sample_rows(w.L, w.P, 32, seed=1)
    parts = []
    for a, b in zip(cu[:-1], cu[1:]):
        sel = sorted({a, b - 1} | {i for i in picked if a <= i < b})
        sl = slice(a, b)
        parts.append(_fwd_sample(q[None, sl], k[None, sl], v[None, sl], out[None, sl],
                                 lse[None, sl], [i - a for i in sel], [4, 17], True))
    samples["lm_varlen_causal"] = SegmentsSample(parts)
    del q, k, v, out, lse

    # backward of the headline workload (dq, dk, dv): algorithmic FLOPs are 2.5x the
    # forward's (five D-length products per visible pair)
    w = LM
    q, k, v = (t.to(dev) for t in make_workload_inputs(w, seed=0))
    do = torch.randn(q.shape, device=dev, generator=g).to(torch.bfloat16)
    out, lse = cea.ring_attn_fwd(q, k, v, P=w.P, causal=True)
    ws = torch.empty(w.B * w.L * w.H, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    f = lambda: cea.ring_attn_bwd(q, k, v, out, lse, do, P=w.P, causal=True, dq=dq, dk=dk, dv=dv,
                                  workspace=ws, stream=stream)
    f()
    ms = _time_loop(f, 3, stream) / 3
    fl = 2.5 * attention_flops(w.B, w.L, w.H, w.D, True)
    res["lm_backward"] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                          "frac": fl / (ms * 1e-3) / 1e12 / peak,
                          "note": "row dots + dK/dV kernel + dQ kernel; 2.5x forward FLOPs"}
    brows = sample_rows(w.L, w.P, 12, seed=2)
    bidx = torch.tensor(brows, device=dev)
    samples["lm_backward"] = DqSample(*(_host(t[:, :, [3, 26]]) for t in (q, k, v, do)), brows,
                                      _host(dq[:, bidx][:, :, [3, 26]]), True)
    del q, k, v, do, out, lse, ws, dq, dk, dv

    # backward with grouped key/value heads: 32 query heads over 8 key/value heads at the
    # headline length (same algorithmic FLOPs as the plain backward of 32 heads)
    q = torch.randn(w.B, w.L, w.H, w.D, device=dev, generator=g).to(torch.bfloat16)
    k, v = (torch.randn(w.B, w.L, 8, w.D, device=dev, generator=g).to(torch.bfloat16)
            for _ in range(2))
    do = torch.randn(q.shape, device=dev, generator=g).to(torch.bfloat16)
    out, lse = cea.ring_attn_fwd_gqa(q, k, v, P=w.P, causal=True)
    ws = torch.empty(w.B * w.L * w.H, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    f = lambda: cea.ring_attn_bwd_gqa(q, k, v, out, lse, do, P=w.P, causal=True, dq=dq, dk=dk,
                                      dv=dv, workspace=ws, stream=stream)
    f()
    ms = _time_loop(f, 3, stream) / 3
    res["lm_gqa_backward"] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                              "frac": fl / (ms * 1e-3) / 1e12 / peak,
                              "note": "32 query heads over 8 key/value heads; 2.5x forward FLOPs"}
    # query heads 3 and 26 read key/value heads 0 and 6
    samples["lm_gqa_backward"] = DqSample(_host(q[:, :, [3, 26]]), _host(k[:, :, [0, 6]]),
                                          _host(v[:, :, [0, 6]]), _host(do[:, :, [3, 26]]), brows,
                                          _host(dq[:, bidx][:, :, [3, 26]]), True)
    del q, k, v, do, out, lse, ws, dq, dk, dv

    # backward over zigzag shards (same causal problem and FLOPs as the plain backward)
    q, k, v, do = (torch.randn(w.B, w.L, w.H, w.D, device=dev, generator=g).to(torch.bfloat16)
                   for _ in range(4))
    out, lse = cea.ring_attn_fwd_zigzag(q, k, v, P=w.P)
    ws = torch.empty(w.B * w.L * w.H, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    f = lambda: cea.ring_attn_bwd_zigzag(q, k, v, out, lse, do, P=w.P, dq=dq, dk=dk, dv=dv,
                                         workspace=ws, stream=stream)
    f()
    ms = _time_loop(f, 3, stream) / 3
    fl = 2.5 * attention_flops(w.B, w.L, w.H, w.D, True)
    res["lm_zigzag_backward"] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                                 "frac": fl / (ms * 1e-3) / 1e12 / peak,
                                 "note": "zigzag shards; 2.5x forward FLOPs"}
    samples["lm_zigzag_backward"] = DqSample(*(_host(t[:, inv][:, :, [3, 26]]) for t in (q, k, v, do)),
                                             brows, _host(dq[:, inv][:, bidx][:, :, [3, 26]]), True)
    del q, k, v, do, out, lse, ws, dq, dk, dv

    # backward of the packed sequences of the forward row above (same lengths)
    q, k, v, do = (torch.randn(w.L, w.H, w.D, device=dev, generator=g).to(torch.bfloat16)
                   for _ in range(4))
    out, lse = cea.ring_attn_fwd_varlen(q, k, v, cu_d, P=w.P, causal=True)
    ws = torch.empty(w.L * w.H, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    def f():
        sched = cea.varlen_schedule(cu_d, w.L, w.P, True, stream=stream)
        cea.ring_attn_bwd_varlen(q, k, v, out, lse, do, cu_d, P=w.P, causal=True, dq=dq, dk=dk,
                                 dv=dv, workspace=ws, stream=stream, schedule=sched)
    f()
    ms = _time_loop(f, 5, stream) / 5
    fl = 2.5 * sum(attention_flops(1, n, w.H, w.D, True) for n in lengths)
    res["lm_varlen_backward"] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                                 "frac": fl / (ms * 1e-3) / 1e12 / peak, "n_seqs": len(lengths),
                                 "note": "packed sequences of the forward row; 2.5x forward "
                                         "FLOPs; schedule computed in each step"}
    parts = []
    for a, b in zip(cu[:-1], cu[1:]):
        sel = sorted({b - 1} | {i for i in brows if a <= i < b})
        sl = slice(a, b)
        sidx = torch.tensor(sel, device=dev)
        parts.append(DqSample(*(_host(t[None, sl][:, :, [3, 26]]) for t in (q, k, v, do)),
                              [i - a for i in sel], _host(dq[None, sidx][:, :, [3, 26]]), True))
    samples["lm_varlen_backward"] = SegmentsSample(parts)
    del q, k, v, do, out, lse, ws, dq, dk, dv, cu_d

    # long-context causal
    w = LONG
    q, k, v = (torch.randn(w.B, w.L, w.H, w.D, device=dev, generator=g).to(torch.bfloat16)
               for _ in range(3))
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.L, w.H), dtype=torch.float32, device=dev)
    f = lambda: cea.ring_attn_fwd(q, k, v, P=w.P, causal=True, out=out, lse=lse, stream=stream)
    f()
    ms = _time_loop(f, 3, stream) / 3
    fl = attention_flops(w.B, w.L, w.H, w.D, True)
    res["long_causal"] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                          "frac": fl / (ms * 1e-3) / 1e12 / peak}
    samples["long_causal"] = _fwd_sample(q, k, v, out, lse, sample_rows(w.L, w.P, 16, seed=1),
                                         [1, 6], True)
    del q, k, v, out, lse
    if cea.check_status(stream) != 0:
        raise RuntimeError("kernel reported a device-side timeout in the secondary rows")
    return res


def run_profile_backward(args):
    """The backward of the causal-LM workload with 8 heads (the small case for profiler
    captures of the row-dot, dK/dV and dQ kernels): `warmup` + `steps` calls, one line out."""
    import context_exact_attention_gb300 as cea

    dev = torch.device("cuda", 0)
    cea.load_library()
    w = dataclasses.replace(LM, H=8)
    q, k, v = (t.to(dev) for t in make_workload_inputs(w, seed=0))
    g = torch.Generator(device=dev).manual_seed(9)
    do = torch.randn(q.shape, device=dev, generator=g).to(torch.bfloat16)
    stream = torch.cuda.current_stream(dev)
    out, lse = cea.ring_attn_fwd(q, k, v, P=w.P, causal=True, stream=stream)
    ws = torch.empty(w.B * w.L * w.H, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    f = lambda: cea.ring_attn_bwd(q, k, v, out, lse, do, P=w.P, causal=True, dq=dq, dk=dk, dv=dv,
                                  workspace=ws, stream=stream)
    for _ in range(args.warmup):
        f()
    ms = _time_loop(f, args.steps, stream) / args.steps
    if cea.check_status(stream) != 0:
        raise RuntimeError("kernel reported a device-side timeout")
    fl = 2.5 * attention_flops(w.B, w.L, w.H, w.D, True)
    print(json.dumps({"case": "causal LM backward, B1 H8 L32768 D128 P8 bf16", "ms": ms,
                      "tflops": fl / (ms * 1e-3) / 1e12}), flush=True)


def packed_lengths(L):
    """The packed-sequence workload's lengths: U[256, 8192) from a CPU generator seeded
    with 5, drawn until they reach L (the last one cut).  Returns (lengths, cu_seqlens)."""
    gl = torch.Generator().manual_seed(5)
    lengths = []
    while sum(lengths) < L:
        lengths.append(int(torch.randint(256, 8192, (1,), generator=gl)))
    lengths[-1] -= sum(lengths) - L
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    return lengths, cu


def run_profile_packed(args):
    """The packed-sequence workload alone (the lm_varlen rows' lengths, H=32, D=128, P=8,
    causal, with a schedule), for profiler captures of the dynamic persistent kernels:
    `warmup` + `steps` forward calls, then `warmup` + `steps` backward calls, one line out."""
    import context_exact_attention_gb300 as cea

    dev = torch.device("cuda", 0)
    cea.load_library()
    stream = torch.cuda.current_stream(dev)
    w = LM
    lengths, cu = packed_lengths(w.L)
    cu_d = torch.tensor(cu, dtype=torch.int32, device=dev)
    g = torch.Generator(device=dev).manual_seed(0)
    q, k, v, do = (torch.randn(w.L, w.H, w.D, device=dev, generator=g).to(torch.bfloat16)
                   for _ in range(4))
    sched = cea.varlen_schedule(cu_d, w.L, w.P, True, stream=stream)
    out = torch.empty_like(q)
    lse = torch.empty((w.L, w.H), dtype=torch.float32, device=dev)
    fwd = lambda: cea.ring_attn_fwd_varlen(q, k, v, cu_d, P=w.P, causal=True, out=out, lse=lse,
                                           stream=stream, schedule=sched)
    for _ in range(args.warmup):
        fwd()
    ms_f = _time_loop(fwd, args.steps, stream) / args.steps
    ws = torch.empty(w.L * w.H, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    bwd = lambda: cea.ring_attn_bwd_varlen(q, k, v, out, lse, do, cu_d, P=w.P, causal=True,
                                           dq=dq, dk=dk, dv=dv, workspace=ws, stream=stream,
                                           schedule=sched)
    for _ in range(args.warmup):
        bwd()
    ms_b = _time_loop(bwd, args.steps, stream) / args.steps
    if cea.check_status(stream) != 0:
        raise RuntimeError("kernel reported a device-side timeout")
    fl = sum(attention_flops(1, n, w.H, w.D, True) for n in lengths)
    print(json.dumps({"case": f"packed sequences {lengths}, H32 D128 P8 bf16, causal",
                      "forward_ms": ms_f, "forward_tflops": fl / (ms_f * 1e-3) / 1e12,
                      "backward_ms": ms_b, "backward_tflops": 2.5 * fl / (ms_b * 1e-3) / 1e12}),
          flush=True)


def run_profile_zigzag(args):
    """The causal-LM zigzag workload with 8 heads (B=1, L=32768, D=128, P=8; inputs above
    L2 at 201 MB), for profiler captures of the zigzag pair-of-SMs kernels: `warmup` +
    `steps` forward calls, then as many backward calls, one line out."""
    import context_exact_attention_gb300 as cea

    dev = torch.device("cuda", 0)
    cea.load_library()
    stream = torch.cuda.current_stream(dev)
    w = LM
    H = 8
    g = torch.Generator(device=dev).manual_seed(0)
    q, k, v, do = (torch.randn(w.B, w.L, H, w.D, device=dev, generator=g).to(torch.bfloat16)
                   for _ in range(4))
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.L, H), dtype=torch.float32, device=dev)
    fwd = lambda: cea.ring_attn_fwd_zigzag(q, k, v, P=w.P, out=out, lse=lse, stream=stream)
    for _ in range(args.warmup):
        fwd()
    ms_f = _time_loop(fwd, args.steps, stream) / args.steps
    ws = torch.empty(w.B * w.L * H, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    bwd = lambda: cea.ring_attn_bwd_zigzag(q, k, v, out, lse, do, P=w.P, dq=dq, dk=dk, dv=dv,
                                           workspace=ws, stream=stream)
    for _ in range(args.warmup):
        bwd()
    ms_b = _time_loop(bwd, args.steps, stream) / args.steps
    if cea.check_status(stream) != 0:
        raise RuntimeError("kernel reported a device-side timeout")
    fl = attention_flops(w.B, w.L, H, w.D, True)
    print(json.dumps({"case": "zigzag shards, B1 H8 L32768 D128 P8 bf16, causal",
                      "forward_ms": ms_f, "forward_tflops": fl / (ms_f * 1e-3) / 1e12,
                      "backward_ms": ms_b, "backward_tflops": 2.5 * fl / (ms_b * 1e-3) / 1e12}),
          flush=True)


def run_profile_hbm(args):
    """The HBM-stream kernels alone, for profiler captures: the LSE merge at the causal-LM
    size (1,048,576 rows x 128, bf16) and the two Ulysses transposes at the Ulysses size
    (B=2, L=8192, H=32, D=128, P=8).  `warmup` rounds of the three, then `steps` calls of
    each kernel in turn (merge, seq2head, head2seq), one JSON line out."""
    import context_exact_attention_gb300 as cea

    dev = torch.device("cuda", 0)
    cea.load_library()
    stream = torch.cuda.current_stream(dev)
    g = torch.Generator(device=dev).manual_seed(0)
    rows, D = LM.B * LM.L * LM.H, LM.D
    oa, ob = (torch.randn(rows, D, device=dev, generator=g).to(torch.bfloat16) for _ in range(2))
    la, lb = (torch.randn(rows, device=dev, generator=g) for _ in range(2))
    oo, lo = torch.empty_like(oa), torch.empty_like(la)
    w = ULYSSES
    x = torch.randn(w.P, w.B, w.L // w.P, w.H, w.D, device=dev, generator=g).to(torch.bfloat16)
    y = torch.empty(w.P, w.B, w.L, w.H // w.P, w.D, device=dev, dtype=torch.bfloat16)
    calls = {
        "merge": (lambda: cea.attn_merge_partials(oa, la, ob, lb, o_out=oo, lse_out=lo,
                                                  stream=stream), rows * (3 * D * 2 + 3 * 4)),
        "seq2head": (lambda: cea.ulysses_seq2head(x, w.P, out=y, stream=stream), 4 * x.numel()),
        "head2seq": (lambda: cea.ulysses_head2seq(y, w.P, out=x, stream=stream), 4 * x.numel()),
    }
    for _ in range(args.warmup):
        for f, _ in calls.values():
            f()
    res = {"case": "merge at causal-LM size; Ulysses transposes at B2 L8192 H32 D128 P8"}
    for name, (f, by) in calls.items():
        ms = _time_loop(f, args.steps, stream) / args.steps
        res[name] = {"ms": ms, "GB/s": by / (ms * 1e-3) / 1e9, "bytes": by}
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-rows", action="store_true", help="skip the secondary measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    ap.add_argument("--sustained-s", type=float, default=2.0,
                    help="seconds of the sustained loop after the headline loop (0: skip)")
    ap.add_argument("--acc-rows", type=int, default=32,
                    help="sampled query rows (all heads) of the headline accuracy check")
    ap.add_argument("--profile-case", action="store_true",
                    help="headline workload with 8 heads instead of 32 (201 MB of inputs, "
                         "still larger than L2): the small case for profiler captures")
    ap.add_argument("--profile-backward", action="store_true",
                    help="only the backward of the headline workload with 8 heads (profiler case)")
    ap.add_argument("--profile-packed", action="store_true",
                    help="only the packed-sequence forward and backward (profiler case)")
    ap.add_argument("--profile-zigzag", action="store_true",
                    help="only the zigzag forward and backward with 8 heads (profiler case)")
    ap.add_argument("--profile-hbm", action="store_true",
                    help="only the merge and Ulysses transpose kernels (profiler case)")
    ap.add_argument("--ref-rows", type=int, default=8,
                    help="query rows (all heads) per reference step")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = _rank_env()
    if world != args.gpus and "RANK" in os.environ:
        print(f"warning: WORLD_SIZE={world} but --gpus {args.gpus}", file=sys.stderr)
    if args.profile_backward:
        run_profile_backward(args)
    elif args.profile_hbm:
        run_profile_hbm(args)
    elif args.profile_packed:
        run_profile_packed(args)
    elif args.profile_zigzag:
        run_profile_zigzag(args)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
