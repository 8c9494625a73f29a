#!/usr/bin/env python3
"""Benchmark: FP32 SGEMM TFLOP/s at M = N = K = 4096 on GB300, and its fraction
of the chip's FP32 FFMA peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--algo ID]

One step is one call of the library (C = alpha*A@B + beta*C) on one batch of
synthetic inputs (uniform[-1, 1), seed of the workload) already resident in
HBM.  Input sets are rotated (at least three, and together more than 1.2x
the L2) so that consecutive steps never find their operands in L2.  Prints
ONE JSON line on rank 0: the headline workload (4096^3 by default) with its
roofline, end-to-end value, oracle baseline and run-to-run spread, and under
"workloads" the other four workloads of the benchmark set (128^3, 1024^3,
4095 x 4097 x 1023 with alpha 0.5 / beta 0.25, 8192^3), each measured the
same way.

Under torchrun (N > 1) every rank multiplies its own copy of the workload on
its own GPU (independent replicas, no data exchange); the host-side barrier
and the max over ranks of the timed region give the whole-job number.

--impl reference times the fp64 CPU oracle on this machine's host cores on a
bounded sample of the same workload (whole output rows), with the same
metric and unit.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fp32_sgemm_gb300 import inputs  # noqa: E402

FFMA_PER_CLK_PER_SM = 128          # FP32 lanes per SM (4 sub-partitions x 32)
PAGES_BEST_TFLOPS = 9.66           # best kernel of the pages at 4096^3 (RTX 3060, "09 Staged")
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "sgemm_ffma_4096_traffic.txt")
TENSOR_PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "sgemm_tf32x3_4096_traffic.txt")
# A kernel's code (the FFMA kernel with every tile configuration; the
# tensor-core kernel); how it is launched is checked separately against the
# plan recorded beside the traffic figure.
# Sources the profiled FFMA launch is built from (configuration 28, the
# automatic choice at 4096^3 with beta == 0): a new configuration file does
# not change it.
KERNEL_SOURCES = ["fp32_sgemm_gb300/csrc/sgemm_ffma.cuh", "fp32_sgemm_gb300/csrc/ptx.cuh",
                  "fp32_sgemm_gb300/csrc/sgemm_algo28.cu"]
TENSOR_KERNEL_SOURCES = ["fp32_sgemm_gb300/csrc/sgemm_tf32x3.cu", "fp32_sgemm_gb300/csrc/ptx.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="sgemm_4096",
                    choices=sorted(inputs.WORKLOADS) + sorted(inputs.EXTRA_WORKLOADS))
    ap.add_argument("--algo", type=int, default=0, help="tile configuration (0 = automatic)")
    ap.add_argument("--math", type=int, default=0,
                    help="0 FP32 FFMA (CUDA cores), 1 error-compensated 3xTF32 (tensor cores)")
    ap.add_argument("--schedule", type=int, default=0,
                    help="0 automatic, 1 whole tiles per CTA, 2 stream-K")
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--tensor-steps", type=int, default=100,
                    help="steps of the 3xTF32 path reported beside the FFMA line (0 = skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="measure only the headline workload (not the other four of the set)")
    ap.add_argument("--repeats", type=int, default=5,
                    help="repeats of the timed K-step loop for the run-to-run spread")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle sample")
    return ap.parse_args()


def kernel_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    if sources is None:
        sources = KERNEL_SOURCES
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(rel.encode())
            h.update(f.read())
    return h.hexdigest()


def plan_signature(plan: dict) -> str:
    return (f"tile {plan['tile_m']}x{plan['tile_n']}x{plan['tile_k']} stages {plan['stages']} "
            f"ctas {plan['ctas']} stream_k {plan['stream_k']} raster_group {plan['raster_group']}")


def profiled_traffic(plan: dict, summary: str = PROFILE_SUMMARY, sources=None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources and the same launch plan; else None."""
    try:
        fields = {}
        for line in open(summary):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
        if fields.get("kernel_source_sha256") != kernel_source_hash(sources):
            return None
        if fields.get("plan") != plan_signature(plan):
            return None
        return float(fields["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm),
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons)}


def sm_max_mhz_query(index: int) -> float | None:
    try:
        out = subprocess.run(["nvidia-smi", f"--id={index}", "--query-gpu=clocks.max.sm",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True,
                             timeout=20).stdout.strip()
        return float(out.splitlines()[0])
    except Exception:
        return None


def measured_hbm():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "of measured (STREAM-style copy)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "of fallback (6.8 TB/s)"


def measure_tf32_peak(dev) -> float | None:
    """Dense TF32 tensor throughput of this GPU, measured in this run: the
    best of 10 cuBLAS TF32 products at 8192^3 through torch (a reference
    figure for the roofline only; nothing of the library runs here)."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    try:
        torch.backends.cuda.matmul.allow_tf32 = True
        n = 8192
        a = torch.rand(n, n, device=dev)
        b = torch.rand(n, n, device=dev)
        c = torch.empty(n, n, device=dev)
        for _ in range(3):
            torch.matmul(a, b, out=c)
        best = None
        for _ in range(10):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        del a, b, c
        torch.cuda.empty_cache()
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except Exception:
        return None
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def tensor_roofline(flops: float, kernel_ms: float, tf32_peak: float | None = None) -> dict:
    """Roofline of the 3xTF32 main kernel: three TF32 products per useful
    multiply-add, against the dense TF32 peak -- measured in this run (cuBLAS
    TF32 at 8192^3) when given, else the measured bf16 tensor peak times the
    nominal TF32/bf16 ratio 1.1/2.25.  useful_frac: the useful FP32 FLOPs
    (2MNK) per second of the kernel over that same peak."""
    if tf32_peak:
        peak = tf32_peak
        basis = "of measured (cuBLAS TF32 8192^3 in this run, best of 10)"
    else:
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                bf16 = float(json.load(f)["bf16_tflops"])
            basis = "of measured (bf16 burst x nominal tf32/bf16 1.1/2.25)"
        except (OSError, KeyError, ValueError):
            bf16 = 1900.0
            basis = "of fallback (1.9 PFLOP/s bf16 x nominal tf32/bf16 1.1/2.25)"
        peak = bf16 * 1.1 / 2.25
    achieved = 3.0 * flops / (kernel_ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": None, "peak_basis": basis,
            "achieved_basis": "3 TF32 MMAs per useful FMA (hi*hi, hi*lo, lo*hi); split pre-pass excluded",
            "useful_frac": achieved / 3.0 / peak}


# ---------------------------------------------------------------- CPU oracle

def oracle_rows_sample(w, p, seconds: float, steps: int = 1, threads: int = 0):
    """Time the oracle on whole output rows of the workload.  Returns
    (flops_per_step, seconds_per_step, rows, threads) for a sample sized so
    that `steps` samples take about `seconds` in total.  threads 0: all the
    host cores OpenMP sees."""
    import oracle
    threads = threads or oracle.max_threads()
    probe_rows = max(1, min(w.M, 32))
    t0 = time.perf_counter()
    oracle.sgemm_ref(probe_rows, w.N, w.K, w.alpha, p.A[:probe_rows], p.B, w.beta,
                     p.C0[:probe_rows] if p.C0 is not None else None, threads=threads)
    rate = probe_rows / max(time.perf_counter() - t0, 1e-6)      # rows per second
    rows = int(max(1, min(w.M, rate * seconds / max(steps, 1))))
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.sgemm_ref(rows, w.N, w.K, w.alpha, p.A[:rows], p.B, w.beta,
                         p.C0[:rows] if p.C0 is not None else None, threads=threads)
        times.append(time.perf_counter() - t0)
    return 2.0 * rows * w.N * w.K, times, rows, threads


def oracle_extra_timings(w, p, seconds: float) -> dict:
    """Oracle timings beside the all-core row sample: single-threaded as well
    for workloads up to 1024^3, and the sampled-entry check the 8192^3
    workload uses (its full-matrix time stated as an extrapolation)."""
    import oracle
    out = {}
    if w.M * w.N * w.K <= 1024 ** 3:
        f, t, rows, _ = oracle_rows_sample(w, p, seconds, 1, threads=1)
        out["single_thread"] = {"value": f / t[0] / 1e12, "unit": "TFLOP/s", "cores": 1,
                                "sample": f"{rows} of {w.M} output rows in {t[0]:.2f} s"}
    if w.samples:
        rows, cols = inputs.sample_entries(w.M, w.N, w.samples, w.seed)
        t0 = time.perf_counter()
        oracle.sgemm_ref_entries(w.K, w.alpha, p.A, p.B, rows, cols, w.beta, p.C0)
        t = time.perf_counter() - t0
        out["sampled_entries"] = {
            "entries": int(w.samples), "seconds": t,
            "value": 2.0 * w.samples * w.K / t / 1e12, "unit": "TFLOP/s",
            "full_matrix_seconds_extrapolated": t * w.M * w.N / w.samples}
    return out


def run_reference(args, w, rank: int, world: int):
    if rank != 0:
        return
    p = inputs.workload_problem(w, "uniform")
    steps = max(1, args.steps)
    warm = max(0, args.warmup)
    budget = 120.0        # seconds for the whole --steps/--warmup run
    flops, times, rows, threads = oracle_rows_sample(w, p, budget, steps + warm)
    timed = times[warm:] if len(times) > warm else times
    t = sum(timed) / len(timed)
    value = flops / t / 1e12
    sample = (f"{rows} of {w.M} output rows per step (all {w.N} columns, K={w.K}), "
              f"fp64 oracle, {threads} threads")
    line = {
        "impl": "reference",
        "metric": "SGEMM TFLOP/s at M=N=K=4096 FP32; % of GB300 FP32 FFMA peak",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": len(timed),
        "warmup": warm, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": value / PAGES_BEST_TFLOPS, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, "cpu oracle sample"),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(w, l2_note: str) -> dict:
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "alpha": w.alpha,
            "beta": w.beta, "seed": w.seed, "layout": "row-major A[M,K] B[K,N] C[M,N]",
            "inputs": "uniform[-1,1) SplitMix64", "l2": l2_note}


# ------------------------------------------------------------------ GPU path

def max_over_ranks(value: float, device) -> float:
    """The largest per-rank value over the process group (a job takes as long
    as its slowest rank); the value itself without a group of several."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's work over the slowest rank's time."""
    return flops_per_rank_step * world / (ms_per_step * 1e-3) / 1e12


class GpuContext:
    """What every measurement on this rank shares: device, stream, handle."""

    def __init__(self, args, rank: int, world: int, local_rank: int):
        import torch
        import fp32_sgemm_gb300 as sg
        self.torch, self.sg = torch, sg
        self.args, self.rank, self.world, self.local_rank = args, rank, world, local_rank
        torch.cuda.set_device(local_rank)
        self.dev = torch.device("cuda", local_rank)
        sg.load_library(build_if_missing=True)
        self.handle = sg.Handle(self.dev)
        self.handle.set_algo(args.algo)
        self.handle.set_schedule(args.schedule)
        self.handle.set_math_mode(args.math)
        props = torch.cuda.get_device_properties(self.dev)
        self.sms = props.multi_processor_count
        self.l2_bytes = getattr(props, "L2_cache_size", 0) or 0
        self.stream = torch.cuda.current_stream(self.dev)
        self.dist = None
        if world > 1:
            import torch.distributed as dist
            self.dist = dist


class WorkloadRun:
    """Device-resident inputs of one workload, rotated over enough sets that
    consecutive steps never find their operands in L2, and the timed loops
    over them."""

    def __init__(self, ctx: GpuContext, w):
        torch = ctx.torch
        self.ctx, self.w = ctx, w
        self.p = inputs.workload_problem(w, "uniform")
        p = self.p
        self.set_bytes = 4 * (p.A.size + p.B.size + w.M * w.N)
        # At least three sets, and together more than 1.2x the L2 (small
        # workloads would otherwise run from L2 between steps).
        want = int(np.ceil(1.2 * max(ctx.l2_bytes, 1) / self.set_bytes)) + 1
        self.nsets = max(3, min(want, 1024))
        A0 = torch.from_numpy(p.A).to(ctx.dev)
        B0 = torch.from_numpy(p.B).to(ctx.dev)
        C0 = (torch.from_numpy(p.C0).to(ctx.dev) if p.C0 is not None
              else torch.zeros((w.M, w.N), device=ctx.dev))
        self.sets = [(A0, B0, C0)] + [(A0.clone(), B0.clone(), C0.clone()) for _ in range(self.nsets - 1)]
        self.ensure_workspace()
        self.plan = ctx.handle.plan(A0, B0, C0, w.alpha, w.beta)

    def ensure_workspace(self):
        A0, B0, _ = self.sets[0]
        h = self.ctx.handle
        h._ensure_workspace(h.workspace_size(self.w.M, self.w.N, self.w.K, A0.data_ptr(), A0.stride(0),
                                             B0.data_ptr(), B0.stride(0)))

    def l2_note(self) -> str:
        return (f"{self.nsets} rotating input sets of {self.set_bytes / 1e6:.1f} MB "
                f"({self.nsets * self.set_bytes / 1e6:.0f} MB > {self.ctx.l2_bytes / 1e6:.0f} MB L2)")

    def timed_loop(self, steps: int, warmup: int, sample_clocks: bool, kernel_events: bool):
        """Warm up, then time `steps` calls on the device (events on the
        launching stream); with kernel_events, also each call's main kernel
        alone (events the library records right around that launch; their
        host cost would count in the step time of small products, so the
        step time comes from a loop without them)."""
        ctx, w = self.ctx, self.w
        torch, h, stream = ctx.torch, ctx.handle, ctx.stream
        for i in range(max(warmup, 3)):
            A, B, C = self.sets[i % self.nsets]
            h.gemm(A, B, C, w.alpha, w.beta, stream=stream)
        torch.cuda.synchronize(ctx.dev)
        assert h.device_error() == 0
        kstart = [torch.cuda.Event(enable_timing=True) for _ in range(steps)] if kernel_events else []
        kstop = [torch.cuda.Event(enable_timing=True) for _ in range(steps)] if kernel_events else []
        for e in kstart + kstop:
            e.record(stream)          # torch creates the event on first record
        torch.cuda.synchronize(ctx.dev)
        if ctx.dist is not None:
            ctx.dist.barrier()
        torch.cuda.synchronize(ctx.dev)
        sampler = ClockSampler(ctx.local_rank) if sample_clocks else None
        if sampler:
            sampler.start()
            time.sleep(0.3)
        t_begin = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_begin.record(stream)
        for i in range(steps):
            A, B, C = self.sets[i % self.nsets]
            if kernel_events:
                h.set_kernel_events(kstart[i], kstop[i])
            h.gemm(A, B, C, w.alpha, w.beta, stream=stream)
        t_end.record(stream)
        torch.cuda.synchronize(ctx.dev)
        h.set_kernel_events(None, None)
        clocks = sampler.stop() if sampler else None
        if ctx.dist is not None:
            ctx.dist.barrier()
        elapsed = t_begin.elapsed_time(t_end)
        kms = [a.elapsed_time(b) for a, b in zip(kstart, kstop)]
        assert h.device_error() == 0
        elapsed = max_over_ranks(elapsed, ctx.dev)
        return elapsed, kms, clocks

    def roofline(self, launch_ms: list, clocks: dict | None) -> dict:
        ctx, w = self.ctx, self.w
        flops = 2.0 * w.M * w.N * w.K
        mean_launch_ms = statistics.mean(launch_ms)
        achieved = flops / (mean_launch_ms * 1e-3) / 1e12
        max_mhz = (clocks or {}).get("sm_max_mhz") or sm_max_mhz_query(ctx.local_rank) or 2070.0
        sus_mhz = (clocks or {}).get("sm_mhz")
        algo_bytes = 4.0 * (w.M * w.K + w.K * w.N + w.M * w.N * (2 if w.beta != 0.0 else 1))
        hbm_peak, hbm_basis = measured_hbm()
        ffma_peak_est = ctx.sms * FFMA_PER_CLK_PER_SM * 2 * max_mhz * 1e6
        if flops / algo_bytes < ffma_peak_est / (hbm_peak * 1e9):
            # Skinny shapes: below the ridge, HBM bounds the kernel.
            gbs = algo_bytes / (mean_launch_ms * 1e-3) / 1e9
            r = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                 "frac": gbs / hbm_peak, "traffic": None, "peak_basis": hbm_basis,
                 "achieved_basis": "compulsory bytes 4(MK+KN+MN) per call over the timed kernels "
                                   "(streaming kernel + split reduction)",
                 "tflops": achieved}
        elif ctx.args.math == 0:
            # Roofline of the dominant (main) kernel: bound by the FP32 FMA pipes.
            peak = ctx.sms * FFMA_PER_CLK_PER_SM * 2 * max_mhz * 1e6 / 1e12
            peak_sus = ctx.sms * FFMA_PER_CLK_PER_SM * 2 * sus_mhz * 1e6 / 1e12 if sus_mhz else None
            r = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                 "frac": achieved / peak,
                 "traffic": profiled_traffic(self.plan) if w.name == "sgemm_4096" else None,
                 "peak_basis": f"{ctx.sms} SMs x {FFMA_PER_CLK_PER_SM} FP32 FMA/clk x 2 FLOP x "
                               f"{max_mhz:.0f} MHz (max SM clock)",
                 "frac_at_sustained_clock": (achieved / peak_sus) if peak_sus else None,
                 "sustained_sm_mhz": sus_mhz}
        else:
            r = tensor_roofline(flops, mean_launch_ms)
        r.update({"kernel_ms_mean": mean_launch_ms, "kernel_ms_min": min(launch_ms),
                  "kernel_ms_median": statistics.median(launch_ms)})
        return r

    def e2e(self, steps: int) -> dict:
        """The same metric through the host-buffer C entry point: pinned host
        A, B (C), copies up, product, copy of C down, all timed."""
        ctx, w, p = self.ctx, self.w, self.p
        torch, sg = ctx.torch, ctx.sg
        Ah = torch.from_numpy(p.A).pin_memory()
        Bh = torch.from_numpy(p.B).pin_memory()
        Ch = (torch.from_numpy(p.C0.copy()) if p.C0 is not None
              else torch.zeros((w.M, w.N))).pin_memory()
        ws = torch.empty(sg.host_workspace_size(w.M, w.N, w.K), dtype=torch.uint8, device=ctx.dev)
        for _ in range(3):
            sg.sgemm_host(Ah, Bh, Ch, w.alpha, w.beta, workspace=ws, handle=ctx.handle, stream=ctx.stream)
        torch.cuda.synchronize(ctx.dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(ctx.stream)
        for _ in range(steps):
            sg.sgemm_host(Ah, Bh, Ch, w.alpha, w.beta, workspace=ws, handle=ctx.handle, stream=ctx.stream)
        e1.record(ctx.stream)
        torch.cuda.synchronize(ctx.dev)
        e_ms = max_over_ranks(e0.elapsed_time(e1) / steps, ctx.dev)
        del ws
        h2d = 4 * (w.M * w.K + w.K * w.N + (w.M * w.N if w.beta != 0.0 else 0))
        return {"value": job_tflops(2.0 * w.M * w.N * w.K, ctx.world, e_ms), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4 * w.M * w.N,
                "ms_per_step": e_ms, "steps": steps,
                "path": "sgemmHostEx: pinned host A,B -> device, SGEMM, C -> pinned host"}

    def cpu_baseline(self, seconds: float) -> dict:
        w, p = self.w, self.p
        c_flops, c_times, rows, threads = oracle_rows_sample(w, p, seconds, 1)
        cpu = {"value": c_flops / c_times[0] / 1e12, "unit": "TFLOP/s", "cores": threads,
               "kind": "oracle",
               "sample": f"{rows} of {w.M} output rows (all {w.N} columns, K={w.K}) "
                         f"in {c_times[0]:.2f} s, fp64 C oracle"}
        cpu.update(oracle_extra_timings(w, p, min(seconds, 10.0)))
        return cpu

    def release(self):
        self.sets = None
        self.ctx.torch.cuda.empty_cache()


def steps_for(run: WorkloadRun, asked: int, min_ms: float = 40.0, cap: int = 4000) -> int:
    """At least the steps asked for, and enough for about min_ms of timed
    work (a 128^3 step takes microseconds)."""
    w = run.w
    est_ms = max(2.0 * w.M * w.N * w.K / 60e12 * 1e3, 0.004)
    return int(min(cap, max(asked, np.ceil(min_ms / est_ms))))


def measure_workload(ctx: GpuContext, w, steps: int, warmup: int, e2e_steps: int, cpu_seconds: float):
    """One entry of the `workloads` map: device throughput, kernel-event
    times and roofline, end-to-end value and the oracle on the host cores."""
    run = WorkloadRun(ctx, w)
    steps = steps_for(run, steps)
    el, _, clocks = run.timed_loop(steps, warmup, True, False)
    _, kms, _ = run.timed_loop(steps, warmup, False, True)
    ms = el / steps
    entry = {
        "value": job_tflops(2.0 * w.M * w.N * w.K, ctx.world, ms), "unit": "TFLOP/s", "ms_per_step": ms,
        "steps": steps, "warmup": max(warmup, 3),
        "config": dict(workload_config(w, run.l2_note()),
                       schedule="stream-K" if run.plan["stream_k"] else "whole tiles",
                       kind=run.plan["kind"],
                       tile=f"{run.plan['tile_m']}x{run.plan['tile_n']}x{run.plan['tile_k']}",
                       ctas=run.plan["ctas"], launches_per_step=run.plan["launches"]),
        "roofline": run.roofline(kms, clocks),
        "gpu_launches": steps * run.plan["launches"],
        "clocks": clocks,
    }
    if w.name == "sgemm_128":
        entry["us_per_step"] = ms * 1e3
    run.release()
    if e2e_steps > 0:
        entry["e2e"] = run.e2e(e2e_steps)
    if ctx.rank == 0 and cpu_seconds > 0:
        entry["cpu_baseline"] = run.cpu_baseline(cpu_seconds)
    return entry


def run_ours(args, w, rank: int, world: int, local_rank: int):
    ctx = GpuContext(args, rank, world, local_rank)
    handle = ctx.handle
    run = WorkloadRun(ctx, w)
    plan = run.plan

    # The step time (value) from a loop with nothing but the calls, clocks
    # sampled meanwhile; the main kernel's own time (roofline) from a second
    # loop with the library's kernel events.
    elapsed_ms, _, clocks = run.timed_loop(args.steps, args.warmup, True, False)
    _, launch_ms, _ = run.timed_loop(args.steps, args.warmup, False, True)

    flops = 2.0 * w.M * w.N * w.K
    ms_per_step = elapsed_ms / args.steps
    value = job_tflops(flops, world, ms_per_step)
    roofline = run.roofline(launch_ms, clocks)

    # Run-to-run spread: the same K-step loop repeated, (max - min) / median
    # of the per-repeat throughput.
    spread = None
    if args.repeats > 1:
        vals = [value]
        for _ in range(args.repeats - 1):
            el, _, _ = run.timed_loop(args.steps, args.warmup, False, False)
            vals.append(job_tflops(flops, world, el / args.steps))
        med = statistics.median(vals)
        spread = {"repeats": len(vals), "steps_each": args.steps, "values": vals,
                  "min": min(vals), "max": max(vals), "median": med,
                  "rel_spread": (max(vals) - min(vals)) / med,
                  "what": "(max - min) / median of the TFLOP/s of repeated K-step loops"}

    # The tensor-core 3xTF32 path on the same inputs (reported beside the
    # FFMA headline, which the metric defines against the FFMA peak).
    tensor_path = None
    if args.math == 0 and args.tensor_steps > 0:
        tf32_peak = measure_tf32_peak(ctx.dev)
        handle.set_math_mode(1)
        run.ensure_workspace()
        tplan = handle.plan(*run.sets[0], w.alpha, w.beta)
        t_el, _, _ = run.timed_loop(args.tensor_steps, args.warmup, False, False)
        _, t_k, _ = run.timed_loop(args.tensor_steps, args.warmup, False, True)
        handle.set_math_mode(0)
        t_step = t_el / args.tensor_steps
        tensor_path = {
            "math": "3xTF32 (tcgen05, error-compensated; same FP32 acceptance bound)",
            "value": job_tflops(flops, world, t_step), "unit": "TFLOP/s",
            "ms_per_step": t_step, "steps": args.tensor_steps,
            "launches_per_step": tplan["launches"],
            "roofline": tensor_roofline(flops, statistics.mean(t_k), tf32_peak),
            "useful_frac_per_call": (job_tflops(flops, world, t_step) / world) / tf32_peak if tf32_peak else None,
            "config": {"tile": f"{tplan['tile_m']}x{tplan['tile_n']}x{tplan['tile_k']}",
                       "schedule": "stream-K" if tplan["stream_k"] else "whole tiles",
                       "ctas": tplan["ctas"]},
        }
        tensor_path["roofline"]["kernel_ms_mean"] = statistics.mean(t_k)
        if w.name == "sgemm_4096":
            tensor_path["roofline"]["traffic"] = profiled_traffic(tplan, TENSOR_PROFILE_SUMMARY,
                                                                  TENSOR_KERNEL_SOURCES)
    config = dict(workload_config(w, run.l2_note()), algo=args.algo,
                  schedule="stream-K" if plan["stream_k"] else "whole tiles",
                  tile=f"{plan['tile_m']}x{plan['tile_n']}x{plan['tile_k']}",
                  stages=plan["stages"], ctas=plan["ctas"], parallelism=f"replicas x{world}")
    run.release()

    e2e = run.e2e(args.e2e_steps) if args.e2e_steps > 0 else None
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = run.cpu_baseline(args.cpu_seconds)

    # The other workloads of the benchmark set, each measured the same way
    # (parity for all of them is checked by the GPU tests).
    workloads = None
    if not args.no_workloads and w.name == "sgemm_4096":
        workloads = {}
        for name in ("sgemm_128", "sgemm_1024", "sgemm_4095x4097x1023", "sgemm_8192"):
            ow = inputs.WORKLOADS[name]
            workloads[name] = measure_workload(
                ctx, ow, args.steps, args.warmup, min(args.e2e_steps, 10 if ow.M >= 8192 else 40),
                0.0 if args.no_cpu_baseline else min(args.cpu_seconds, 6.0))

    if rank != 0:
        return
    line = {
        "metric": "SGEMM TFLOP/s at M=N=K=4096 FP32; % of GB300 FP32 FFMA peak",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": value / PAGES_BEST_TFLOPS,
        "vs_baseline_ref": "9.66 TFLOP/s: the pages' best kernel at 4096^3 on an RTX 3060",
        "dtype": "f32", "data": "synthetic",
        "config": config,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "spread": spread,
        "tensor_path": tensor_path,
        "workloads": workloads,
        "gpu_launches": args.steps * plan["launches"],
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    w = inputs.WORKLOADS.get(args.workload) or inputs.EXTRA_WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
