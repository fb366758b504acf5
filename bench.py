#!/usr/bin/env python3
"""Benchmark of the GB300 GEMM library.

Default workload (one step = one gemm_run through the C ABI): the dense bf16
GEMM M = N = K = 4096, A row-major, B col-major, entries N(0,1)/sqrt(K),
C bf16 N(0,1), alpha 1.5, beta 0.5, bf16 D, fp32 accumulation.  Metric:
TFLOP/s = 2*M*N*K / time.  Three rotating input sets (384 MB) keep the
operands out of the 129 MB L2 between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config c2|c1|c3m1|c3m16|c3m64|c4|c5|c2f8]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the GEMM has no exchange step), timing is the max over ranks and the value
is the total work of all ranks divided by it.  ``--impl reference`` times the
CPU oracle (the only reference this project has) on a bounded sample.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---- multi-rank aggregation -----------------------------------------------------------

def max_over_ranks(ms, dist, device="cuda"):
    """The largest of the ranks' timings (every rank gets it); `ms` itself
    when there is no process group."""
    if dist is None:
        return float(ms)
    import torch

    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(unit_per_step, steps, world, ms):
    """Whole-job throughput: every rank runs `steps` steps of `unit_per_step`
    units each; the job takes the slowest rank's `ms`."""
    return world * unit_per_step * steps / (ms / 1e3)


# ---- workloads ----------------------------------------------------------------------

WORKLOADS = {
    "c1": dict(desc="dense fp16 GEMM M=N=K=256, fp32 D, alpha 1 beta 0", kind="dense"),
    "c2": dict(desc="dense bf16 GEMM M=N=K=4096, A row-major, B col-major, N(0,1)/sqrt(K), C bf16 N(0,1), "
                    "alpha 1.5 beta 0.5, bf16 D", kind="dense"),
    "c3m1": dict(desc="decode bf16 GEMM M=1 N=4096 K=14336, N(0,0.02), bf16 D", kind="dense", M=1),
    "c3m16": dict(desc="decode bf16 GEMM M=16 N=4096 K=14336, N(0,0.02), bf16 D", kind="dense", M=16),
    "c3m64": dict(desc="decode bf16 GEMM M=64 N=4096 K=14336, N(0,0.02), bf16 D", kind="dense", M=64),
    "c4": dict(desc="W4A16 GEMM M=128 K=4096 N=11008, int4 B + fp16 group-128 scales, bf16 D", kind="dense"),
    "c5": dict(desc="grouped MoE bf16 GEMM, 8 experts, 4096 tokens Zipf(1.2), K=4096, N=14336, bf16 D",
               kind="grouped"),
    "c2f8": dict(desc="dense E4M3 GEMM M=N=K=4096, A row-major, B col-major, N(0,1) rounded to E4M3, C bf16 "
                      "N(0,1), alpha 1.5/64 beta 0.5, bf16 D", kind="dense"),
}


def register_shape(shape):
    """Add a dense bf16 workload of the given "M,N,K" with C2's recipe; returns its name."""
    M, N, K = (int(x) for x in shape.split(","))
    if min(M, N, K) < 1:
        raise ValueError(f"bad shape {shape!r}")
    cfg = f"dense{M}x{N}x{K}"
    WORKLOADS[cfg] = dict(desc=f"dense bf16 GEMM M={M} N={N} K={K}, A row-major, B col-major, N(0,1)/sqrt(K), "
                               f"C bf16 N(0,1), alpha 1.5 beta 0.5, bf16 D", kind="dense", shape=(M, N, K))
    return cfg


def make_problem(cfg):
    if "shape" in WORKLOADS.get(cfg, {}):
        M, N, K = WORKLOADS[cfg]["shape"]
        return synth.config2(M=M, N=N, K=K)
    if cfg == "c1":
        return synth.config1()
    if cfg == "c2":
        return synth.config2()
    if cfg.startswith("c3m"):
        return synth.config3(int(cfg[3:]))
    if cfg == "c4":
        return synth.config4()
    if cfg == "c5":
        return synth.config5()
    if cfg == "c2f8":
        return synth.config2_fp8()
    raise ValueError(cfg)


def flops_of(p):
    if hasattr(p, "counts"):
        return 2.0 * int(p.offsets[-1]) * p.N * p.K
    return 2.0 * p.M * p.N * p.K


def algorithmic_bytes(p):
    """A, B (packed for int4), U/V, C (if beta != 0) and D, each once."""
    if hasattr(p, "counts"):
        T = int(p.offsets[-1])
        experts = int((p.counts > 0).sum())
        return 2 * (T * p.K + experts * p.N * p.K + T * p.N)
    out_b = 4 if p.d_type == synth.F32 else 2
    in_b = 1 if p.a_type in (synth.E4M3, synth.E5M2) else 2
    b = in_b * p.M * p.K + out_b * p.M * p.N
    b += p.N * p.K // 2 if p.b_type == synth.S4 else in_b * p.N * p.K
    if p.V is not None:
        b += p.V.size * (4 if p.v_type == synth.F32 else 2)
    if p.beta != 0.0:
        b += out_b * p.M * p.N
    return b


def metric_of(cfg):
    """(metric, unit, bound) per workload: HBM-bound ones report GB/s."""
    if cfg.startswith("c3"):
        return "GEMM HBM GB/s (decode)", "GB/s", "hbm"
    return "GEMM TFLOP/s", "TFLOP/s", "tensor"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(files=None):
    """Hash of the kernel sources a profile was taken on: the listed files of
    the package's csrc/ (all of them when none are listed)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_gemm_tcgen05_gb300", "csrc")
    if files is None:
        files = sorted(f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    for f in files:
        path = os.path.join(csrc, f)
        if not os.path.exists(path):
            return None
        with open(path, "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def profile_traffic(cfg, choice):
    """Per-launch DRAM bytes from the committed ncu summary of this workload,
    or None when it is missing, was taken on other kernel sources, or on
    another kernel choice than the one this run dispatched."""
    import glob
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", f"*_{cfg}.md"))):
        text = open(path).read()
        m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
        s = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
        f = re.search(r"kernel_sources:\s*(.+)", text)
        files = f.group(1).split() if f else None
        c = re.search(r"kernel_choice:\s*(\S+)", text)
        if not m or not s or s.group(1) != kernel_source_hash(files):
            continue
        if c and c.group(1) != choice:
            continue
        return float(m.group(1))
    return None


# ---- clocks -------------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples, kept for a time window."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [r for t, r in self.rows if t0 <= t <= t1 + 0.1]
        if not rows:
            rows = [r for _, r in self.rows[-3:]]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[2]) for r in rows if len(r) > 3 and r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if len(r) > 3 and r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for i, n in enumerate(names):
                if len(r) > 6 + i and r[6 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---- our implementation ---------------------------------------------------------------

class Runner:
    """Device buffers plus pre-built ctypes arguments for repeated gemm_run calls."""

    def __init__(self, p, sets, qg, torch, splitk=0, streamk=0):
        self.p, self.qg, self.torch = p, qg, torch
        self.h = qg.gemm_create()
        self.ws = qg.Workspace()
        self.op = qg.gemm_op_t(0, 0, 0, p.gb if getattr(p, "V", None) is not None else 0, splitk, streamk)
        self.stream = qg.current_stream()
        self.grouped = hasattr(p, "counts")
        self.args = []
        self.bufs = []
        for s in range(sets):
            self.args.append(self._build(s))

    def _dev(self, bits, dtype):
        torch = self.torch
        if dtype == synth.S4:
            return torch.from_numpy(np.ascontiguousarray(bits)).cuda()
        if dtype == synth.F32:
            return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.float32)).cuda()
        if dtype in (synth.E4M3, synth.E5M2):
            f8 = torch.float8_e4m3fn if dtype == synth.E4M3 else torch.float8_e5m2
            return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).view(f8).cuda()
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
        return t.view(torch.bfloat16 if dtype == synth.BF16 else torch.float16).cuda()

    def _build(self, s):
        qg, torch, p = self.qg, self.torch, self.p
        if self.grouped:
            A, B = self._dev(p.A, p.a_type), self._dev(p.B, p.a_type)
            off = torch.from_numpy(p.offsets.astype(np.int32)).cuda()
            T = int(p.offsets[-1])
            D = torch.empty(T, p.N, dtype=torch.bfloat16, device="cuda")
            self.bufs.append((A, B, off, D))
            return dict(A=A, B=B, off=off, D=D, Ad=qg.row_major(A), Bd=qg.col_major_from_nk(B), Dd=qg.row_major(D))
        A = self._dev(p.A, p.a_type)
        B = self._dev(p.B, p.b_type)
        dt = {synth.F32: torch.float32, synth.F16: torch.float16, synth.BF16: torch.bfloat16}[p.d_type]
        D = torch.empty(p.M, p.N, dtype=dt, device="cuda")
        C = self._dev(p.C, p.c_type) if p.beta != 0.0 else None
        V = self._dev(p.V, p.v_type) if p.V is not None else None
        self.bufs.append((A, B, C, D, V))
        d = dict(A=A, B=B, C=C, D=D, V=V, Ad=qg.row_major(A), Bd=qg.col_major_from_nk(B, k=p.K, type_=p.b_type),
                 Dd=qg.row_major(D), Cd=qg.row_major(C) if C is not None else None,
                 Vd=qg.layout(p.v_type, qg.GEMM_ROW_MAJOR, p.K // p.gb, p.N, p.N) if V is not None else None)
        return d

    def run(self, s, stream=None):
        qg, p, a = self.qg, self.p, self.args[s]
        st = stream if stream is not None else self.stream
        if self.grouped:
            rc = qg.gemm_run_grouped(self.h, self.op, p.alpha, a["A"].data_ptr(), a["Ad"], None, None,
                                     a["B"].data_ptr(), a["Bd"], None, None, p.beta, None, None, a["D"].data_ptr(),
                                     a["Dd"], a["off"].data_ptr(), len(p.counts), self.ws.c, st)
        else:
            rc = qg.gemm_run(self.h, self.op, p.alpha, a["A"].data_ptr(), a["Ad"], None, None, a["B"].data_ptr(),
                             a["Bd"], qg.ptr(a["V"]), a["Vd"], p.beta, qg.ptr(a["C"]), a["Cd"], a["D"].data_ptr(),
                             a["Dd"], self.ws.c, st)
        if rc:
            raise RuntimeError(f"gemm_run failed: {qg.gemm_status_string(rc)}")


def input_sets(cfg, one_set):
    """Rotating copies of the inputs so that consecutive steps do not find
    their operands in the 129 MB L2: at least 3 x L2 in total (at most 8)."""
    if cfg == "c2":
        return 3
    return max(1, min(8, int(np.ceil(3 * 129e6 / max(one_set, 1)))))


def time_steps(R, sets, steps, launch, torch, qg, barrier, soak_s=0.0):
    """Time exactly `steps` calls of R.run on the current stream.

    graph: the calls are captured once into a CUDA graph (as an engine
    replaying its layers would), replayed untimed (for at least soak_s seconds,
    so clock samples see the load), then timed as one replay.  eager: one
    gemm_run per step with CUDA events around every launch.  Returns
    (total_ms, per-launch ms or None, t0, t1) with t0/t1 the wall-clock window
    of the untimed soak plus the timed region."""
    stream = torch.cuda.current_stream()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if launch == "graph":
        cap = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=cap):
            for i in range(steps):
                R.run(i % sets, qg.current_stream())
        torch.cuda.synchronize()
        t0 = time.time()
        graph.replay()
        torch.cuda.synchronize()
        while time.time() - t0 < soak_s:
            graph.replay()
            torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        start.record(stream)
        graph.replay()
        end.record(stream)
        torch.cuda.synchronize()
        barrier()
        t1 = time.time()
        del graph
        return start.elapsed_time(end), None, t0, t1
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(stream)
    for i in range(steps):
        evs[i][0].record(stream)
        R.run(i % sets)
        evs[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    t1 = time.time()
    return start.elapsed_time(end), [a.elapsed_time(b) for a, b in evs], t0, t1


def roofline_of(cfg, p, avg_launch_s, traffic, peaks, peak_src):
    """The roofline object for one workload: achieved algorithmic bytes or
    flops per launch over the launch's duration, against the measured peak."""
    flops, abytes = flops_of(p), algorithmic_bytes(p)
    _, _, bound = metric_of(cfg)
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    if bound == "hbm":
        achieved, peak, r_unit = abytes / avg_launch_s / 1e9, hbm_peak, "GB/s"
    else:
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])) * tensor_peak_ratio(p)
        achieved, r_unit = flops / avg_launch_s / 1e12, "TFLOP/s"
    r = {"bound": bound, "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": r_unit,
         "frac": round(achieved / peak, 4), "traffic": traffic,
         "peak_source": f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})"
                        + ("" if tensor_peak_ratio(p) == 1 else f" x {tensor_peak_ratio(p):g} (nominal dense ratio of "
                                                                  f"this input type to bf16)"),
         "algorithmic_per_launch": abytes if bound == "hbm" else flops,
         "avg_launch_us": round(avg_launch_s * 1e6, 3)}
    if bound == "tensor":
        r["hbm_gbs"] = round(abytes / avg_launch_s / 1e9, 1)
        r["hbm_frac"] = round(abytes / avg_launch_s / 1e9 / hbm_peak, 4)
        r["min_roofline_us"] = round(max(flops / (peak * 1e12), abytes / (hbm_peak * 1e9)) * 1e6, 3)
        r["min_roofline_frac"] = round(r["min_roofline_us"] / (avg_launch_s * 1e6), 4)
    return r


def tensor_peak_ratio(p):
    """Nominal dense tensor rate of the problem's input type relative to bf16
    (fp8: 4.5 / 2.25 PFLOP/s)."""
    return 2.0 if getattr(p, "a_type", None) in (synth.E4M3, synth.E5M2) else 1.0


SCHEDULES = {"auto": (0, 0), "unsplit": (1, 0), "splitk8": (8, 0), "streamk": (0, 1)}

# Workloads measured beside the headline, each in the same process: the
# decode shapes under every schedule the decode workload names, plus the
# automatic choice.
SUB_CONFIGS = ([("c1", "auto")] +
               [(f"c3m{m}", s) for m in (1, 16, 64) for s in ("auto", "unsplit", "splitk8", "streamk")] +
               [("c4", "auto"), ("c5", "auto"), ("c2f8", "auto")])


def measure_config(cfg, sched, steps, warmup, launch, sampler, peaks, peak_src, qg, torch, p=None):
    """One workload under one schedule, timed like the headline; returns its
    entry of the "configs" object."""
    p = make_problem(cfg) if p is None else p
    metric, unit, bound = metric_of(cfg)
    abytes, flops = algorithmic_bytes(p), flops_of(p)
    sets = input_sets(cfg, abytes)
    splitk, streamk = SCHEDULES[sched]
    R = Runner(p, sets, qg, torch, splitk=splitk, streamk=streamk)
    try:
        for i in range(warmup):
            R.run(i % sets)
        torch.cuda.synchronize()
        if qg.gemm_device_status(R.h, R.stream):
            raise RuntimeError(f"{cfg}/{sched}: device status reported a timeout during warm-up")
        choice = qg.gemm_last_choice(R.h)
        total_ms, launch_ms, t0, t1 = time_steps(R, sets, steps, launch, torch, qg, lambda: None, soak_s=0.2)
        if qg.gemm_device_status(R.h, R.stream):
            raise RuntimeError(f"{cfg}/{sched}: device status reported a timeout")
    finally:
        qg.gemm_destroy(R.h)
    avg_launch_s = (statistics.mean(launch_ms) if launch_ms else total_ms / steps) / 1e3
    unit_per_step = abytes / 1e9 if unit == "GB/s" else flops / 1e12
    traffic = profile_traffic(cfg, choice)
    entry = {"workload": WORKLOADS[cfg]["desc"], "schedule": sched, "kernel": choice, "metric": metric,
             "value": round(job_throughput(unit_per_step, steps, 1, total_ms), 3), "unit": unit,
             "steps": steps, "ms_per_step": round(total_ms / steps, 5), "gpu_launches": steps,
             "roofline": roofline_of(cfg, p, avg_launch_s, traffic, peaks, peak_src),
             "clocks": sampler.summary(t0, t1)}
    del R
    torch.cuda.empty_cache()
    return entry


def run_ours(args, rank, world, cfg):
    import torch

    import quantized_gemm_tcgen05_gb300 as qg

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    p = make_problem(cfg)
    flops = flops_of(p)
    abytes = algorithmic_bytes(p)
    metric, unit, bound = metric_of(cfg)
    unit_per_step = abytes / 1e9 if unit == "GB/s" else flops / 1e12
    one_set = abytes
    sets = input_sets(cfg, one_set)
    R = Runner(p, sets, qg, torch)

    def barrier():
        if dist is not None:
            dist.barrier()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(1.5)  # nvidia-smi needs a moment before its first sample
    for i in range(args.warmup):
        R.run(i % sets)
    torch.cuda.synchronize()
    if qg.gemm_device_status(R.h, R.stream):
        raise RuntimeError("device status reported a timeout during warm-up")
    choice = qg.gemm_last_choice(R.h)

    # timed region: exactly K steps (see time_steps)
    total_ms, launch_ms, t0, t1 = time_steps(R, sets, args.steps, args.launch, torch, qg, barrier, soak_s=0.3)
    clocks = sampler.summary(t0, t1)
    total_ms = max_over_ranks(total_ms, dist)
    ms_per_step = total_ms / args.steps
    value = job_throughput(unit_per_step, args.steps, world, total_ms)
    if qg.gemm_device_status(R.h, R.stream):
        raise RuntimeError("device status reported a timeout during the timed region")

    # end-to-end through the C ABI with host buffers: H2D of this step's
    # inputs from pinned memory, the GEMM, D2H of the result, every step
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(R, torch, unit_per_step, unit, world, dist, steps=max(3, min(20, args.steps)))

    peaks, peak_src = load_peaks()
    # per-launch duration: the event pair around each launch (eager), or the
    # graph replay divided by its launches (back-to-back kernels, so this also
    # charges the inter-kernel gaps to the kernel: a conservative figure)
    avg_launch_s = (statistics.mean(launch_ms) if launch_ms else ms_per_step) / 1e3
    traffic = profile_traffic(cfg, choice)
    line = {
        "metric": metric, "value": round(value, 3), "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": synth.DTYPE_NAMES.get(p.a_type, "bf16"),
        "data": "synthetic (seeded, shapes and distributions of the workload)",
        "config": {"workload": WORKLOADS[cfg]["desc"], "kernel": choice, "parallelism": f"replicas x{world}",
                   "launch": "CUDA graph of the K gemm_run calls" if args.launch == "graph" else "eager gemm_run per step",
                   "l2": f"{sets} rotating input sets ({sets * one_set / 1e6:.0f} MB) so operands are not L2-resident"},
        "roofline": roofline_of(cfg, p, avg_launch_s, traffic, peaks, peak_src),
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": args.steps,
    }
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(p, cfg, unit)
    R.qg.gemm_destroy(R.h)
    del R
    torch.cuda.empty_cache()
    # the other workloads, one process, after the headline (one GPU only)
    if world == 1 and not args.no_configs:
        sub_steps = max(3, min(20, args.steps))
        configs = {}
        made = {}
        for c, s in SUB_CONFIGS:
            if c == cfg and s == "auto":
                continue
            if c not in made:
                made.clear()
                made[c] = make_problem(c)
            key = c if s == "auto" else f"{c}/{s}"
            configs[key] = measure_config(c, s, sub_steps, 3, args.launch, sampler, peaks, peak_src, qg, torch,
                                          p=made[c])
        line["configs"] = configs
    sampler.stop()
    if dist is not None:
        dist.destroy_process_group()
    return line


def measure_e2e(R, torch, unit_per_step, unit, world, dist, steps):
    stream = torch.cuda.current_stream()
    a = R.args[0]
    host = {}
    h2d = 0
    names = ["A", "B", "C", "V", "off"] if not R.grouped else ["A", "B", "off"]
    for n in names:
        t = a.get(n)
        if t is None:
            continue
        host[n] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        host[n].copy_(t)
        h2d += t.numel() * t.element_size()
    D = a["D"]
    hD = torch.empty(D.shape, dtype=D.dtype, pin_memory=True)
    d2h = D.numel() * D.element_size()
    torch.cuda.synchronize()

    def step():
        for n, h in host.items():
            a[n].copy_(h, non_blocking=True)
        R.run(0)
        hD.copy_(D, non_blocking=True)

    step()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    s.record(stream)
    for _ in range(steps):
        step()
    e.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(s.elapsed_time(e), dist)
    return {"value": round(job_throughput(unit_per_step, steps, world, ms), 3), "unit": unit,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms / steps, 4)}


# ---- the CPU oracle as baseline / reference arm ---------------------------------------------

def oracle_sample(p, rows):
    """The first `rows` rows of the problem (all columns, full K) -- a bounded
    sample for the CPU oracle."""
    import copy

    if hasattr(p, "counts"):
        e = int(np.argmax(p.counts))
        lo = int(p.offsets[e])
        q = synth.Problem(min(rows, int(p.counts[e])), p.N, p.K, p.a_type, p.a_type, p.d_type,
                          p.A[lo:lo + rows], p.B[e], alpha=p.alpha, beta=p.beta)
        return q
    q = copy.copy(p)
    q.M = min(rows, p.M)
    q.A = p.A[:q.M]
    if p.C is not None:
        q.C = p.C[:q.M]
    return q


def cpu_baseline(p, cfg, unit, target_s=10.0):
    """The oracle on the first rows of the workload, doubling the row count
    until one call takes about target_s (or the whole problem is covered)."""
    import oracle

    full_rows = int(p.counts.max()) if hasattr(p, "counts") else p.M
    rows = 8
    while True:
        q = oracle_sample(p, rows)
        t = time.perf_counter()
        oracle.gemm(q)
        dt = time.perf_counter() - t
        if dt >= target_s or q.M >= full_rows or rows >= 4096:
            break
        rows = min(full_rows, rows * 2 if dt > target_s / 8 else rows * 4)
    f = flops_of(q)
    val = (algorithmic_bytes(q) / dt / 1e9) if unit == "GB/s" else f / dt / 1e12
    return {"value": round(val, 6), "unit": unit, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"first {q.M} rows x all {q.N} columns x full K={q.K} of the workload, "
                      f"{dt:.2f} s of fp64 OpenMP work"}


def run_reference(args, rank, world, cfg):
    import oracle

    if rank != 0:
        return None
    p = make_problem(cfg)
    metric, unit, _ = metric_of(cfg)
    oracle.build()
    rows = 16
    q = oracle_sample(p, rows)
    for _ in range(args.warmup if args.warmup < 3 else 3):
        oracle.gemm(oracle_sample(p, 2))
    times = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.gemm(q)
        times.append(time.perf_counter() - t)
        if time.perf_counter() - t_all > 150:
            break
    dt = statistics.mean(times)
    val = (algorithmic_bytes(q) / dt / 1e9) if unit == "GB/s" else flops_of(q) / dt / 1e12
    sample = f"first {q.M} rows x all {q.N} columns x full K={q.K} per step"
    return {"impl": "reference", "metric": metric, "value": round(val, 6), "unit": unit, "n_gpus": world,
            "steps": len(times), "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOADS[cfg]["desc"], "sample": sample},
            "cpu_baseline": {"value": round(val, 6), "unit": unit, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(val, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=sorted(WORKLOADS), default="c2")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="time only the --config workload")
    ap.add_argument("--launch", choices=["graph", "eager"], default="graph")
    ap.add_argument("--shape", help="M,N,K: a dense bf16 problem of this shape with C2's recipe, instead of --config")
    args = ap.parse_args()
    if args.shape:
        args.config = register_shape(args.shape)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
    if "RANK" not in os.environ:
        world = 1 if args.gpus == 1 else args.gpus
        if world > 1:
            ap.error("run --gpus N > 1 under torchrun (one process per GPU)")
    if args.impl == "reference":
        line = run_reference(args, rank, world, args.config)
    else:
        line = run_ours(args, rank, world, args.config)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
