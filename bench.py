"""Benchmark: FP16 GEMM TFLOPS on GB300 through the gemm_f16 C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload gemm_4096]

One step = one C = A*B of the workload (the whole hot path: tile schedule,
TMA producer ring, tcgen05 MMA, epilogue, and for split workloads the
fixed-order reduction).  The 4096^3 workload rotates through eight seeded A/B
pairs (8 x 64 MiB = 512 MiB, well above the 129 MB L2), so consecutive
steps never find their inputs in L2.  Protocol from the "Xe2 ESIMD GEMM"
page, "Performance testing": random non-zero inputs, rotating buffers, a 5 s
pause, >= 20 warm-up and 1000 timed iterations by default (more when a
step is short, so that the timed region lasts at least 50 ms and the clock
samples fall inside it).

Timing: CUDA events on the launching stream around exactly K steps, with a
barrier and a device synchronise on both sides; max over ranks.  With
torchrun each rank runs an independent replica on its own GPU (the GEMM has
no exchange step, so there is no collective on the data path).

Extra keys: roofline (dominant kernel vs the measured dense 16-bit tensor
peak, or HBM bandwidth: its work per launch over the mean duration of its
launches, timed with CUDA events on its own stream in a second pass of the
timed region's steps; the whole step's figure beside it), cpu_baseline (the FP64 oracle on a bounded row sample, host cores,
with the host's machine type and CPU model), e2e (same metric through
gemm_f16_run_host with pinned host buffers, copies inside the timed region),
clocks (nvidia-smi sampled under load), sustained (the same step re-timed
back to back over >= 0.3 s with its own clock samples, against the measured
sustained tensor peak), gpu_launches (kernels launched in the timed region).

--impl reference times the FP64 CPU oracle on the same workload instead
(bounded row samples per step).

--graph submits the timed steps as replays of a CUDA graph of consecutive
steps captured after the warm-up (the same kernels, no host call per step).

--workload attn_256 / attn_ragged / attn_4096 measures the attention
forward kernel (attn_f16_fwd, head dimension 256) instead: one step = one
O = softmax(Q K^T / 16) V over all batches and heads, TFLOPS counted as
4 * B * H * Sq * Skv * 256.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic_inputs as si  # noqa: E402

METRIC = "FP16 GEMM TFLOPS at M=N=K=4096 on 1 GB300; % of dense FP16 tensor peak"
ATTN_METRIC = "FP16 attention forward TFLOPS, head dim 256, on 1 GB300"
FALLBACK_TENSOR_TFLOPS = 1900.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = [os.path.join(ROOT, "async_barrier_pipelined_gb300", "csrc", f)
                  for f in ("plan.cu", "gemm_f16.cu", "attn_f16.cu", "host.h", "common.cuh",
                            "gemm_pair.cuh", "ptx.cuh", "schedule.h", "attn_f16.cuh",
                            "attn_pair.cuh", "gemm_quad.cuh")]
SUSTAINED_S = 0.3


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 1000, or more when a step is short, so that "
                         "the timed region lasts at least 50 ms and the clock samples cover it)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gemm_4096",
                    choices=sorted(si.WORKLOADS) + sorted(si.ATTN_WORKLOADS))
    ap.add_argument("--sleep", type=float, default=5.0,
                    help="idle seconds before the warm-up (page protocol: 5)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel", type=int, default=0, choices=[0, 1, 2, 3],
                    help="GEMM: 0 automatic, 1 single-CTA kernel, 2 CTA pair 256x256, "
                         "3 cluster of four (two pairs sharing A); "
                         "attention: 0 automatic, 1 single CTA, 2 CTA pair")
    ap.add_argument("--no-sustained", action="store_true",
                    help="skip the sustained (>= 0.3 s) re-timing of the step")
    ap.add_argument("--graph", action="store_true",
                    help="submit the timed steps as replays of a CUDA graph of consecutive "
                         "steps (captured after the warm-up) instead of one host call each: "
                         "the launch-bound small workloads then show the GPU's time")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU seconds for the oracle baseline sample")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers
def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


FALLBACK_HBM_GBS = 6800.0


def load_peaks():
    """(dense 16-bit tensor TFLOP/s burst, sustained, HBM GB/s, source)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            pk = json.load(fh)
        return (float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", 0.0)),
                float(pk["hbm_gbs"]), "measured")
    except Exception:
        return FALLBACK_TENSOR_TFLOPS, 1700.0, FALLBACK_HBM_GBS, "fallback"


def compulsory_bytes(w: si.Workload) -> int:
    """Bytes a GEMM must move at least: read A and B once, write C once (fp16)."""
    return 2 * (w.M * w.K + w.K * w.N + w.M * w.N)


def kernel_bytes(w: si.Workload) -> int:
    """Bytes the product kernel must move at least: read A and B once, then
    write C (fp16), or with split_k > 1 the split_k FP32 partial tiles that
    the reduction kernel adds."""
    out = 4 * w.split_k * w.M * w.N if w.split_k > 1 else 2 * w.M * w.N
    return 2 * (w.M * w.K + w.K * w.N) + out


KERNEL_TIMING_NOTE = ("algorithmic work per launch / the product (or attention) kernel's "
                      "duration per launch, the smaller of two CUDA-event upper bounds: "
                      "kernel_ms_events (events on the launch stream directly around each "
                      "launch, over the timed region's steps run again right after it; the "
                      "event pair also serialises each launch behind the previous kernel) and "
                      "the timed region's step time (all of a step's launches, overlapped); "
                      "step_achieved divides by the step time")


def kernel_duration(kms: float, ms_step: float):
    """(ms per launch, which bound) for the roofline: both the event-pair
    time and the step time bound the kernel's own duration from above."""
    if kms <= ms_step:
        return kms, "kernel events"
    return ms_step, "timed-region step time"


def _traffic_entry(workload: str):
    """The workload's entry of the committed ncu summary, or None when the
    kernel sources changed since it was captured."""
    try:
        with open(TRAFFIC_FILE) as fh:
            e = json.load(fh).get(workload)
        if e and e.get("kernel_source_sha") == kernel_source_hash():
            return e
    except Exception:
        pass
    return None


def load_traffic(workload: str):
    """Per-launch DRAM bytes of the dominant kernel from a committed ncu
    summary, or None when the kernel source changed since it was captured."""
    e = _traffic_entry(workload)
    return float(e["dram_bytes_per_launch"]) if e else None


def load_tensor_pipe(workload: str):
    """The dominant kernel's tensor-pipe activity from a committed `ncu --set
    full` capture ({"of_active_pct", "of_elapsed_pct", "sm_ghz"}; a clock-
    independent measure of how busy the tensor cores are), or None."""
    e = _traffic_entry(workload)
    return e.get("tensor_pipe") if e else None


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons in the background."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.proc = None
        self.tmp = None
        self.marks = {}

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", f"-lms={self.interval}"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark(self, name):
        self.marks[name] = time.time()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = [ln.strip().split(", ") for ln in self.tmp if ln.strip()]
        self.tmp.close()
        os.unlink(self.tmp.name)
        return self._summarise(rows)

    def _summarise(self, rows):
        from datetime import datetime
        t0 = self.marks.get("load_start", 0)
        t1 = self.marks.get("timed_end", time.time())
        under, reasons, smax = [], set(), None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 10:
                continue
            try:
                ts = datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            if not (t0 <= ts <= t1 + 0.05):
                continue
            try:
                sm, smx = float(r[2]), float(r[3])
            except ValueError:
                continue
            smax = smx
            under.append(sm)
            for name, val in zip(names, r[6:10]):
                if val.strip() == "Active":
                    reasons.add(name)
        if not under:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                    "samples": 0,
                    "note": (f"region of {1e3 * (t1 - t0):.1f} ms is shorter than the "
                             f"{self.interval} ms sampling period: no sample fell in it "
                             "(see the sustained record for clocks under load)")}
        return {"sm_mhz": statistics.median(under), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(under),
                "window": "last warm-up steps and the timed region"}


def max_over_ranks(ms: float, world: int, dev=None) -> float:
    """The slowest rank's time: every rank contributes its own event time
    and all receive the maximum (a no-op for one process)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, steps: int, world: int, ms_total: float) -> float:
    """Work of all ranks (each runs `steps` steps of its own replica) over
    the slowest rank's time."""
    return flops_per_step * steps * world / (ms_total * 1e-3) / 1e12


MIN_TIMED_S = 0.05


def auto_steps(step, barrier, stream, world, dev, start, n=50):
    """Timed-step count when none is given: 1000, or as many as fill
    MIN_TIMED_S (at most 200000), from the time of n more untimed steps
    (the slowest rank's, so that every rank runs the same count).
    Returns (steps, n)."""
    import math
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        step(start + i)
    e1.record(stream)
    e1.synchronize()
    barrier()
    per_ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / n
    return int(min(200000, max(1000, math.ceil(MIN_TIMED_S * 1e3 / max(per_ms, 1e-6))))), n


GRAPH_STEPS = 32


def capture_steps(step, stream, first: int, n: int):
    """A CUDA graph of n consecutive steps (first .. first + n - 1), captured
    on `stream` after the warm-up has built every buffer the steps use."""
    import torch
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(n):
            step(first + i)
    return graph


def issue_steps(step, stream, steps: int, graph, gsteps: int):
    """The timed region's work: `steps` host calls, or steps / gsteps
    replays of the captured graph (steps is then a multiple of gsteps)."""
    import torch
    if graph is None:
        for i in range(steps):
            step(i)
        return
    with torch.cuda.stream(stream):
        for _ in range(steps // gsteps):
            graph.replay()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def sustained_record(step, barrier, stream, dev, world, ms_step, flops_per_step, start,
                     peak_sustained, peak_burst):
    """The same step timed again over at least SUSTAINED_S seconds (back to
    back, so that the GPU settles at its power limit), with its own clock
    samples: the figure a long run would see, against the measured
    sustained tensor peak as well as the burst one."""
    import math
    import torch
    n = int(max(1, math.ceil(SUSTAINED_S * 1e3 / max(ms_step, 1e-6))))
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.2)
    sampler.mark("load_start")
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        step(start + i)
    e1.record(stream)
    e1.synchronize()
    barrier()
    sampler.mark("timed_end")
    clocks = sampler.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    value = whole_job_tflops(flops_per_step, n, world, ms)
    return {"value": value, "unit": "TFLOPS", "steps": n, "ms_per_step": ms / n,
            "seconds": ms * 1e-3,
            "frac_of_sustained_peak": value / world / peak_sustained if peak_sustained else None,
            "frac_of_burst_peak": value / world / peak_burst, "clocks": clocks}


def kernel_timing_pass(g, plan, step, barrier, steps: int, start: int, world, dev):
    """Mean duration of the dominant kernel's launches: the timed region's
    steps run once more, right after it, with the library's kernel timing
    records on (a CUDA event pair on the launch stream directly around each
    product / attention kernel launch, read back with gemm_f16_kernel_time).
    A separate pass because an event between two launches stops the next
    kernel's set-up from overlapping the previous kernel (programmatic
    dependent launch), which would slow the step being timed.  Returns
    (ms per launch, max over ranks; launches timed on this rank)."""
    plan.kernel_time()                      # forget earlier records
    plan.set_option(g.OPT_KERNEL_TIMING, 1)
    try:
        for i in range(steps):
            step(start + i)
        barrier()
    finally:
        plan.set_option(g.OPT_KERNEL_TIMING, 0)
    ms, n = plan.kernel_time()
    if n <= 0:
        raise RuntimeError("no kernel launch was timed")
    return max_over_ranks(ms / n, world, dev), n


def host_record() -> dict:
    """Machine and CPU model of the host the CPU baseline ran on."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as fh:
                for ln in fh:
                    if ln.lower().startswith(("model name", "cpu part")):
                        model = ln.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    return {"machine": platform.machine(), "cpu_model": model,
            "logical_cpus": os.cpu_count()}


# ------------------------------------------------------------------ CPU oracle
def cpu_oracle_sample(w: si.Workload, rows: np.ndarray, A_bits, B_bits):
    import oracle
    t0 = time.perf_counter()
    oracle.gemm_f16(A_bits, B_bits, rows=rows)
    return time.perf_counter() - t0


def cpu_baseline(w: si.Workload, target_s: float, pairs_bits):
    """Oracle TFLOPS on a bounded sample of the workload (~target_s seconds).

    If one full product fits the budget, whole products are repeated over
    the workload's pairs until the budget is spent; otherwise an evenly
    spaced subset of the rows of C (pair 0) is computed.
    """
    import oracle
    threads = oracle.num_threads()
    a0, b0 = pairs_bits[0]
    r0 = int(min(w.M, max(threads, 64)))
    t_cal = cpu_oracle_sample(w, np.arange(r0), a0, b0)        # calibration, untimed
    per_row = max(t_cal / r0, 1e-9)
    if per_row * w.M > target_s:
        n = int(max(1, target_s / per_row))
        rows = np.linspace(0, w.M - 1, n).astype(np.int64)
        t = cpu_oracle_sample(w, rows, a0, b0)
        flops = 2.0 * n * w.N * w.K
        sample = (f"{n} of {w.M} rows of C (evenly spaced) for pair 0: "
                  f"{flops / 1e9:.1f} GFLOP in {t:.1f} s, FP64 triple loop")
    else:
        t, flops, products = 0.0, 0.0, 0
        while t < target_s:
            a, b = pairs_bits[products % len(pairs_bits)]
            t += cpu_oracle_sample(w, np.arange(w.M), a, b)
            flops += 2.0 * w.M * w.N * w.K
            products += 1
        sample = (f"{products} full products over {min(products, len(pairs_bits))} "
                  f"pair(s): {flops / 1e9:.1f} GFLOP in {t:.1f} s, FP64 triple loop")
    return {"value": flops / t / 1e12, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
            "sample": sample, "host": host_record()}


# ------------------------------------------------------------------ arms
def attn_oracle_rows(w, b: int, h: int, rows):
    """Seconds for the FP64 oracle on `rows` of head (b, h)."""
    import oracle
    q, k, v = w.head_bits(b, h, rows)
    t0 = time.perf_counter()
    oracle.attention_f16(q, k, v, w.scale)
    return time.perf_counter() - t0


def attn_cpu_baseline(w, target_s: float):
    """Oracle TFLOPS on a bounded sample: evenly spaced query rows of the
    heads (b, h) taken in order until ~target_s seconds are spent."""
    import oracle
    threads = oracle.num_threads()
    r0 = int(min(w.Sq, max(threads, 16)))
    t_cal = attn_oracle_rows(w, 0, 0, np.arange(r0))            # calibration, untimed
    per_row = max(t_cal / r0, 1e-9)
    n = int(max(1, min(w.Sq, target_s / per_row / 4)))
    rows = np.linspace(0, w.Sq - 1, n).astype(np.int64)
    t, done, heads = 0.0, 0, 0
    while t < target_s and heads < w.B * w.H:
        t += attn_oracle_rows(w, heads // w.H, heads % w.H, rows)
        done += n
        heads += 1
    flops = 4.0 * done * w.Skv * w.D
    return {"value": flops / t / 1e12, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
            "sample": f"{n} of {w.Sq} query rows (evenly spaced) of {heads} head(s): "
                      f"{flops / 1e9:.1f} GFLOP in {t:.1f} s, FP64 plain softmax",
            "host": host_record()}


def attn_config(w):
    return {"workload": w.name, "batch": w.B, "heads": w.H, "seq_q": w.Sq, "seq_kv": w.Skv,
            "head_dim": w.D, "scale": w.scale, "mask": "none",
            "layout": "[batch, head, seq, 256] contiguous, binary16",
            "inputs": f"Q, K normal sigma={w.qk_sigma}; V uniform non-zero on [-1, 1]",
            "cache": "inputs larger than L2 (Q, K, V, O %.0f MB)" % (
                2.0 * w.D * w.B * w.H * (2 * w.Sq + 2 * w.Skv) / 1e6)}


def run_reference_attention(args):
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    import oracle
    w = si.ATTN_WORKLOADS[args.workload]
    threads = oracle.num_threads()
    budget = 120.0
    steps = args.steps + args.warmup
    probe = np.arange(min(w.Sq, max(threads, 16)))
    per_row = max(attn_oracle_rows(w, 0, 0, probe) / len(probe), 1e-6)
    n = int(max(1, min(w.Sq, budget / steps / per_row)))
    for i in range(args.warmup):
        attn_oracle_rows(w, 0, i % w.H, (np.arange(n) + i * n) % w.Sq)
    total = 0.0
    for i in range(args.steps):
        hh = i % (w.B * w.H)
        total += attn_oracle_rows(w, hh // w.H, hh % w.H, (np.arange(n) + i * n) % w.Sq)
    flops = 4.0 * n * args.steps * w.Skv * w.D
    value = flops / total / 1e12
    line = {
        "metric": ATTN_METRIC, "value": value, "unit": "TFLOPS", "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": attn_config(w),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                         "sample": f"{n} query rows of one head per step, FP64 plain softmax",
                         "host": host_record()},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args):
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    if args.workload in si.ATTN_WORKLOADS:
        return run_reference_attention(args)
    import oracle
    w = si.WORKLOADS[args.workload]
    A_bits, B_bits = w.pair_bits(0)
    threads = oracle.num_threads()
    budget = 120.0
    steps = args.steps + args.warmup
    # size each step's sample so the whole run ends within ~budget seconds
    probe_rows = np.arange(min(w.M, threads))
    t = cpu_oracle_sample(w, probe_rows, A_bits, B_bits)
    per_row = max(t / len(probe_rows), 1e-6)
    n = int(max(1, min(w.M, budget / steps / per_row)))
    rows_all = np.arange(w.M)
    for i in range(args.warmup):
        cpu_oracle_sample(w, rows_all[(i * n) % w.M:][:n], A_bits, B_bits)
    total = 0.0
    done_rows = 0
    for i in range(args.steps):
        sel = np.roll(rows_all, -((i * n) % w.M))[:n]
        total += cpu_oracle_sample(w, sel, A_bits, B_bits)
        done_rows += n
    flops = 2.0 * done_rows * w.N * w.K
    value = flops / total / 1e12
    ms_per_step = total / args.steps * 1e3
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                         "sample": f"{n} rows of C per step ({n}x{w.N} outputs, "
                                   f"K={w.K}), FP64 triple loop", "host": host_record()},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w: si.Workload):
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "split_k": w.split_k,
            "pairs": len(w.keys), "layout": "row-major A (MxK), B (KxN), C (MxN)",
            "accumulate": "f32", "inputs": f"{w.dist} scale={w.scale} eps={w.eps}",
            "cache": ("rotating A/B pairs larger than L2"
                      if len(w.keys) > 1 else "inputs resident (no rotation)")}


def run_attention(args):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_setup(args)
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import async_barrier_pipelined_gb300 as g
    from async_barrier_pipelined_gb300 import build as gbuild
    gbuild.build()

    w = si.ATTN_WORKLOADS[args.workload]
    qb, kb, vb = w.bits()
    Q, K, V = (torch.from_numpy(x.view(np.float16)).to(dev) for x in (qb, kb, vb))
    O = torch.empty_like(Q)
    stream = torch.cuda.Stream(device=dev)
    plan = g.Plan(dev.index)
    plan.set_option(g.OPT_ATTN_KERNEL, min(args.kernel, 2))
    use_pair = args.kernel != 1
    # key ranges the library picks for this shape: > 1 adds the merging kernel
    ranges = g.attn_f16_key_ranges(plan.handle, w.B, w.H, w.Sq, w.Skv)
    launches_per_step = 1 if ranges == 1 else 2

    npairs = 1   # one set of inputs (a CUDA graph of --graph covers GRAPH_STEPS steps)
    # the C entry point with its arguments marshalled once (as the GEMM steps
    # call gemm_f16_run directly), so host overhead does not pace small cases
    lib = g.load()
    c_st = lambda X: (ctypes.c_int64 * 3)(X.stride(0), X.stride(1), X.stride(2))
    call_args = (plan.handle, w.B, w.H, w.Sq, w.Skv, w.D, Q.data_ptr(), c_st(Q), K.data_ptr(),
                 c_st(K), V.data_ptr(), c_st(V), O.data_ptr(), c_st(O), float(w.scale),
                 int(stream.cuda_stream))

    def step(i):
        rc = lib.attn_f16_fwd(*call_args)
        if rc != 0:
            raise RuntimeError(f"attn_f16_fwd returned {rc}")

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    step(0)
    torch.cuda.synchronize(dev)
    if plan.status() != 0:
        raise RuntimeError("device status error")

    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(args.sleep)
    sampler.mark("load_start")
    for i in range(args.warmup):
        step(i)
    barrier()
    probe = 0
    if args.steps is None:
        args.steps, probe = auto_steps(step, barrier, stream, world, dev, args.warmup)
    graph, gsteps = None, 0
    if args.graph:
        gsteps = GRAPH_STEPS * npairs
        args.steps = (args.steps + gsteps - 1) // gsteps * gsteps
        graph = capture_steps(step, stream, 0, gsteps)
        issue_steps(step, stream, gsteps, graph, gsteps)     # one untimed replay
        barrier()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    issue_steps(step, stream, args.steps, graph, gsteps)
    ev1.record(stream)
    ev1.synchronize()
    barrier()
    sampler.mark("timed_end")
    clocks = sampler.stop()
    ms_total = ev0.elapsed_time(ev1)
    if plan.status() != 0:
        raise RuntimeError("device status error after the timed region")
    ms_total = max_over_ranks(ms_total, world, dev)
    ms_step = ms_total / args.steps
    value = whole_job_tflops(float(w.flops), args.steps, world, ms_total)

    peak, peak_sus, peak_hbm, peak_kind = load_peaks()
    sustained = None
    if not args.no_sustained:
        sustained = sustained_record(step, barrier, stream, dev, world, ms_step, float(w.flops),
                                     args.steps, peak_sus, peak)
        if plan.status() != 0:
            raise RuntimeError("device status error in the sustained region")
    kms_ev, klaunches = kernel_timing_pass(g, plan, step, barrier, args.steps, 0, world, dev)
    if plan.status() != 0:
        raise RuntimeError("device status error in the kernel timing pass")
    kms, kfrom = kernel_duration(kms_ev, ms_step)
    achieved = float(w.flops) / (kms * 1e-3) / 1e12
    step_achieved = float(w.flops) / (ms_step * 1e-3) / 1e12
    cbytes = 2.0 * w.D * w.B * w.H * (2 * w.Sq + 2 * w.Skv)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "kernel_ms_per_launch": kms, "duration_from": kfrom, "kernel_ms_events": kms_ev,
                "kernel_launches_timed": klaunches,
                "step_achieved": step_achieved, "step_frac": step_achieved / peak,
                "achieved_from": KERNEL_TIMING_NOTE,
                "peak_source": f"{peak_kind} dense bf16 burst (fp16 runs at the same rate)",
                "algorithmic_flops_per_launch": float(w.flops),
                "traffic": load_traffic(w.name) if use_pair else None,
                "tensor_pipe_ncu": load_tensor_pipe(w.name) if use_pair else None,
                "flop_per_byte": float(w.flops) / cbytes,
                "kernel": ("gf16::attnp::attn_f16_fwd_pair_kernel" if use_pair
                           else "gf16::attn::attn_f16_fwd_kernel")
                + ("" if ranges == 1 else " + gf16::attnp::attn_combine_kernel")}

    e2e = None
    if not args.no_e2e:
        hq, hk, hv = (torch.from_numpy(x.view(np.float16)).pin_memory() for x in (qb, kb, vb))
        ho = torch.empty(O.shape, dtype=torch.float16).pin_memory()

        def host_step(i):
            g.attention_host(plan, hq, hk, hv, ho, scale=w.scale, stream=stream)

        e2e_steps = max(1, min(args.steps, 20))
        for i in range(3):
            host_step(i)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(e2e_steps):
            host_step(i)
        e1.record(stream)
        e1.synchronize()
        barrier()
        ms_e2e = e0.elapsed_time(e1)
        ms_e2e = max_over_ranks(ms_e2e, world, dev)
        if plan.status() != 0:
            raise RuntimeError("device status error in the e2e region")
        e2e = {"value": whole_job_tflops(float(w.flops), e2e_steps, world, ms_e2e),
               "unit": "TFLOPS", "h2d_bytes_per_step": int(qb.nbytes + kb.nbytes + vb.nbytes),
               "d2h_bytes_per_step": int(qb.nbytes), "steps": e2e_steps,
               "api": "attn_f16_fwd_host (pinned host Q, K, V, O; copies overlap across calls)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = attn_cpu_baseline(w, args.cpu_seconds)
    plan.close()
    if rank == 0:
        line = {
            "metric": ATTN_METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup + probe, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16", "data": "synthetic",
            "config": dict(attn_config(w), kernel=("CTA pair (tcgen05 cta_group::2, 256 query "
                                                   "rows, 128-key blocks)" if use_pair else
                                                   "single CTA (128 query rows, 64-key blocks)"),
                           key_ranges=ranges,
                           submission=(f"CUDA graph of {gsteps} steps, replayed"
                                       if graph is not None else "one host call per step")),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "sustained": sustained,
            "gpu_launches": args.steps * launches_per_step,
            "pct_of_peak": 100.0 * step_achieved / peak,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_ours(args):
    import torch
    import torch.distributed as dist

    if args.workload in si.ATTN_WORKLOADS:
        return run_attention(args)

    world, rank, local = dist_setup(args)
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import async_barrier_pipelined_gb300 as g
    from async_barrier_pipelined_gb300 import build as gbuild
    gbuild.build()

    w = si.WORKLOADS[args.workload]
    npairs = len(w.keys)
    pairs_bits = [w.pair_bits(p) for p in range(npairs)]
    A = [torch.from_numpy(a.view(np.float16)).to(dev) for a, _ in pairs_bits]
    B = [torch.from_numpy(b.view(np.float16)).to(dev) for _, b in pairs_bits]
    C = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sh = int(stream.cuda_stream)
    plan = g.Plan(dev.index)
    plan.set_option(g.OPT_KERNEL, args.kernel)
    # what one call enqueues: kernel choice, launches (product, split
    # reduction, repack of an A whose rows are off 128-byte lines)
    info = g.gemm_f16_run_info(plan.handle, 0, w.M, w.N, w.K, w.K, w.split_k)
    launches_per_step = info["launches"]

    def step(i):
        p = i % npairs
        g.gemm_f16_run(plan.handle, w.M, w.N, w.K, A[p].data_ptr(), w.K, B[p].data_ptr(), w.N,
                       C.data_ptr(), w.N, w.split_k, sh)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # a first call, checked for a device-side timeout before any timing
    step(0)
    torch.cuda.synchronize(dev)
    st = plan.status()
    if st != 0:
        raise RuntimeError(f"device status {st}")

    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(args.sleep)
    sampler.mark("load_start")
    for i in range(args.warmup):
        step(i)
    barrier()
    probe = 0
    if args.steps is None:
        args.steps, probe = auto_steps(step, barrier, stream, world, dev, args.warmup)
    graph, gsteps = None, 0
    if args.graph:
        gsteps = GRAPH_STEPS * npairs
        args.steps = (args.steps + gsteps - 1) // gsteps * gsteps
        graph = capture_steps(step, stream, 0, gsteps)
        issue_steps(step, stream, gsteps, graph, gsteps)     # one untimed replay
        barrier()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    issue_steps(step, stream, args.steps, graph, gsteps)
    ev1.record(stream)
    ev1.synchronize()
    barrier()
    sampler.mark("timed_end")
    clocks = sampler.stop()
    ms_total = ev0.elapsed_time(ev1)
    st = plan.status()
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed region")
    ms_total = max_over_ranks(ms_total, world, dev)
    ms_step = ms_total / args.steps
    value = whole_job_tflops(float(w.flops), args.steps, world, ms_total)

    peak, peak_sus, peak_hbm, peak_kind = load_peaks()
    sustained = None
    if not args.no_sustained:
        sustained = sustained_record(step, barrier, stream, dev, world, ms_step, float(w.flops),
                                     args.steps, peak_sus, peak)
        if plan.status() != 0:
            raise RuntimeError("device status error in the sustained region")
    # Dominant kernel: the product kernel (single-CTA, pair or cluster of
    # four), timed on its own in a second pass of the same steps; the step
    # figures (all of a step's launches: repack, K-halves merge, split
    # reduction) sit beside it.  Bound: tensor if the workload's FLOP per
    # compulsory byte is above the ridge point (tensor peak / HBM
    # bandwidth), else HBM.
    kms_ev, klaunches = kernel_timing_pass(g, plan, step, barrier, args.steps, 0, world, dev)
    if plan.status() != 0:
        raise RuntimeError("device status error in the kernel timing pass")
    kms, kfrom = kernel_duration(kms_ev, ms_step)
    cbytes = compulsory_bytes(w)
    kbytes = kernel_bytes(w)
    ridge = peak * 1e12 / (peak_hbm * 1e9)
    timing = {"kernel_ms_per_launch": kms, "duration_from": kfrom, "kernel_ms_events": kms_ev,
              "kernel_launches_timed": klaunches, "achieved_from": KERNEL_TIMING_NOTE}
    if w.flops / cbytes >= ridge:
        achieved = float(w.flops) / (kms * 1e-3) / 1e12
        step_achieved = float(w.flops) / (ms_step * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak,
                    "peak_source": f"{peak_kind} dense bf16 burst (fp16 runs at the same rate)",
                    "algorithmic_flops_per_launch": float(w.flops), **timing,
                    "step_achieved": step_achieved, "step_frac": step_achieved / peak}
    else:
        achieved = kbytes / (kms * 1e-3) / 1e9
        step_achieved = cbytes / (ms_step * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak_hbm, "unit": "GB/s",
                    "frac": achieved / peak_hbm, "peak_source": f"{peak_kind} HBM copy bandwidth",
                    "algorithmic_bytes_per_launch": float(kbytes), **timing,
                    "step_achieved": step_achieved, "step_frac": step_achieved / peak_hbm,
                    "step_algorithmic_bytes": float(cbytes),
                    "tflops": float(w.flops) / (ms_step * 1e-3) / 1e12}
    roofline["traffic"] = load_traffic(w.name)
    roofline["tensor_pipe_ncu"] = load_tensor_pipe(w.name)
    roofline["flop_per_byte"] = w.flops / cbytes
    roofline["ridge_flop_per_byte"] = ridge

    # e2e through gemm_f16_run_host: pinned host buffers, copies timed
    e2e = None
    if not args.no_e2e:
        hA = [torch.from_numpy(a.view(np.float16)).pin_memory() for a, _ in pairs_bits]
        hB = [torch.from_numpy(b.view(np.float16)).pin_memory() for _, b in pairs_bits]
        hC = torch.empty((w.M, w.N), dtype=torch.float16).pin_memory()

        def host_step(i):
            p = i % npairs
            g.gemm_f16_run_host(plan.handle, w.M, w.N, w.K, hA[p].data_ptr(), w.K,
                                hB[p].data_ptr(), w.N, hC.data_ptr(), w.N, w.split_k, sh)

        e2e_steps = max(1, min(args.steps, 200))
        for i in range(3):
            host_step(i)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(e2e_steps):
            host_step(i)
        e1.record(stream)
        e1.synchronize()
        barrier()
        ms_e2e = e0.elapsed_time(e1)
        ms_e2e = max_over_ranks(ms_e2e, world, dev)
        if plan.status() != 0:
            raise RuntimeError("device status error in the e2e region")
        e2e = {"value": whole_job_tflops(float(w.flops), e2e_steps, world, ms_e2e),
               "unit": "TFLOPS",
               "h2d_bytes_per_step": 2 * (w.M * w.K + w.K * w.N),
               "d2h_bytes_per_step": 2 * w.M * w.N,
               "steps": e2e_steps, "api": "gemm_f16_run_host (pinned host buffers)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds, pairs_bits)

    plan_sms = plan.get_option(g.INFO_NUM_SMS)
    plan_pairs = plan.get_option(g.INFO_MAX_PAIRS)
    plan_quads = plan.get_option(g.INFO_MAX_QUADS)
    kernel_id = info["kernel"]
    kernel_desc = {
        3: "cluster of four (two tcgen05 cta_group::2 pairs sharing A by multicast, "
           "256x512 cluster tiles)",
        2: "CTA pair (tcgen05 cta_group::2, 256x256 tiles)",
    }.get(kernel_id, f"single CTA (tcgen05 cta_group::1, 128x{info['tile_width']} tiles)")
    if info["repack_a"]:
        kernel_desc += "; A repacked to 128-byte-aligned rows first"
    if info["launches"] > 1 + (w.split_k > 1) + info["repack_a"]:
        kernel_desc += "; partial last wave in K halves, merged by a second kernel"
    roofline["kernel"] = {3: "gf16::quad::gemm_f16_quad_kernel",
                          2: "gf16::pair::gemm_f16_pair_kernel"}.get(kernel_id,
                                                                    "gf16::gemm_f16_kernel")
    roofline["launches_per_step"] = launches_per_step
    plan.close()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup + probe, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16", "data": "synthetic",
            "config": dict(workload_config(w), kernel=kernel_desc,
                           sms=plan_sms, max_pairs=plan_pairs,
                           max_quads=plan_quads,
                           submission=(f"CUDA graph of {gsteps} steps, replayed"
                                       if graph is not None else "one host call per step")),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "clocks": clocks, "sustained": sustained,
            "gpu_launches": args.steps * launches_per_step,
            "pct_of_peak": 100.0 * (float(w.flops) / (ms_step * 1e-3) / 1e12) / peak,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        if args.steps is None:
            args.steps = 1000   # each a bounded CPU sample
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
