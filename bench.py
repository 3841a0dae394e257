"""Benchmark of the sm_103a fp16 GEMM (fp32 accumulate) on its headline workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one C = A.B through the library's public API on the square
M = N = K = 8192 workload (seed 5, A and B uniform in [-0.5, 0.5), made on
the host and copied to the device before timing). Rank 0 prints one JSON line.

* value: whole-job TFLOP/s, 2*M*N*K per step per rank, over the max over
  ranks of the device time (CUDA events on the launching stream) of K
  back-to-back steps bracketed by a barrier and a synchronize. A and B
  (256 MiB) and C (128 MiB) exceed the 129 MB L2, so no flush is needed
  (--flush-l2 adds one between steps, outside the timed events).
* roofline: the GEMM kernel's average launch duration from per-launch CUDA
  events, 2*M*N*K flops per launch, against the measured dense bf16 tensor
  peak (fp16 runs at the bf16 rate) from MEASURED_PEAKS.json; traffic is the
  DRAM bytes per launch from the committed ncu summary for this kernel
  source, or null when the kernel changed since that capture.
* e2e: the same metric end to end from pinned host memory: per step the
  host-to-device copies of A and B, the GEMM, and the device-to-host copy of C.
* cpu_baseline: the CPU oracle on a bounded, seeded sample of rows of the
  same workload, timed on this host's cores (rank 0 only).
* --impl reference: the oracle alone as the reference arm, on the host.
Multi-GPU (torchrun): replicas only. Every rank runs the same workload on its
own GPU with no collective on the data path; scaling is weak.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fp16 GEMM TFLOP/s (fp32 acc) at M=N=K=8192; % of GB300 dense fp16 TC peak"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1000 * 1000
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def kernel_source_hash() -> str:
    """Hash of the CUDA sources: identifies the kernel an ncu capture measured."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_fp16_gemm_fp32_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(workload: str, tile: str, group_size_m: int):
    """DRAM bytes per launch recorded by ncu for this kernel source, or None."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(f"{workload}/{tile}/G{group_size_m}")
    if not e or e.get("kernel_hash") != kernel_source_hash():
        return None
    return float(e["dram_bytes_per_launch"])


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.samples = []  # (host time, sm_mhz, max_mhz, power_w, reasons)
        self.proc = None
        self.thread = None
        self.gpu_index = gpu_index
        self.period_ms = period_ms

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            try:
                pw = float(parts[3])
            except ValueError:
                pw = None
            names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            reasons = [n for n, v in zip(names[1:], parts[5:9]) if v.lower().startswith("active")]
            self.samples.append((time.time(), sm, mx, pw, reasons))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed region"
        if not inside and self.samples:
            mid = 0.5 * (t0 + t1)
            inside = sorted(self.samples, key=lambda s: abs(s[0] - mid))[:3]
            window = "nearest samples (timed region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "no samples"}
        reasons = sorted({r for s in inside for r in s[4]})
        pw = [s[3] for s in inside if s[3] is not None]
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": max(s[2] for s in inside),
                "reasons": reasons, "power_w_max": max(pw) if pw else None, "samples": len(inside),
                "window": window}


# ---------------------------------------------------------------- ranks
def max_over_ranks(ms: float, device, world: int) -> float:
    """The slowest rank's time: every rank contributes its own, all receive the max."""
    if world <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Replicas: every rank runs `steps` steps; the job's rate is all ranks' flops
    over the slowest rank's time."""
    return flops_per_step * steps * world / (max_ms * 1e-3) / 1e12


# ---------------------------------------------------------------- CPU oracle
def time_oracle(A, B, rows, nthreads):
    from oracle import gemm as og
    t = time.perf_counter()
    og.gemm_rows(A, B, rows=rows, nthreads=nthreads)
    return time.perf_counter() - t


def cpu_baseline(A, B, seed: int, target_s: float):
    """The oracle as it stands on a seeded sample of rows: ~target_s of work."""
    import numpy as np
    import torch
    from oracle import gemm as og

    M, K = A.shape
    N = B.shape[1]
    cores = og.default_threads()
    g = torch.Generator().manual_seed(seed + 2000)
    perm = torch.randperm(M, generator=g).numpy()
    # two calibration runs separate the per-call cost (B converted to fp32 once
    # per call) from the per-row cost
    calib = min(M, max(cores, 4))
    t1 = time_oracle(A, B, np.sort(perm[:calib]), cores)
    t2 = time_oracle(A, B, np.sort(perm[:2 * calib]), cores) if 2 * calib <= M else 2 * t1
    per_row = max((t2 - t1) / calib, 1e-6)
    fixed = max(t1 - calib * per_row, 0.0)
    n = int(min(M, max(calib, (target_s - fixed) / per_row)))
    rows = np.sort(perm[:n])
    t = time_oracle(A, B, rows, cores)
    flops = 2.0 * n * N * K
    return {"value": flops / t / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} seeded rows of the {M}x{N}x{K} workload ({n * N} outputs), "
                      f"{t:.1f} s, fp32 ascending-k C loop with {cores} threads"}


# ---------------------------------------------------------------- arms
def run_reference(args, w, rank, world):
    """Reference arm: the CPU oracle on the host, bounded samples per step."""
    if rank != 0:
        return 0
    import numpy as np
    import torch
    from dense_fp16_gemm_fp32_gb300 import inputs
    from oracle import gemm as og

    A, B = inputs.gemm_inputs(w.M, w.N, w.K, w.seed)
    cores = og.default_threads()
    g = torch.Generator().manual_seed(w.seed + 3000)
    perm = torch.randperm(w.M, generator=g).numpy()
    calib = min(w.M, max(cores, 4))
    per_row = max(time_oracle(A, B, np.sort(perm[:calib]), cores) / calib, 1e-6)
    budget = args.reference_budget_s
    rows_per_step = int(max(1, min(w.M, budget / max(1, args.steps + args.warmup) / per_row)))
    for i in range(args.warmup):
        time_oracle(A, B, np.sort(perm[:rows_per_step]), cores)
    t = 0.0
    for i in range(args.steps):
        off = (i * rows_per_step) % max(1, w.M - rows_per_step + 1)
        t += time_oracle(A, B, np.sort(perm[off:off + rows_per_step]), cores)
    flops = 2.0 * rows_per_step * w.N * w.K * args.steps
    value = flops / t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": config_dict(w, args, tile=None),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{rows_per_step} seeded rows of {w.M}x{w.N}x{w.K} per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def config_dict(w, args, tile):
    l2 = ("flush: a 256 MiB buffer is written between timed steps" if args.flush_l2 else
          "inputs larger than L2: A+B = %d MiB, C = %d MiB vs 129 MB L2; no flush"
          % ((2 * w.M * w.K + 2 * w.K * w.N) >> 20, (2 * w.M * w.N) >> 20))
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "seed": w.seed,
            "inputs": "A,B = torch.rand(fp16, host generator seeded) - 0.5",
            "accumulate": "f32", "output": "f16, rounded once", "tile": tile,
            "group_size_m": args.group_size_m, "l2": l2, "parallelism": "replicas"}


def run_ours(args, w, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import dense_fp16_gemm_fp32_gb300 as g
    from dense_fp16_gemm_fp32_gb300 import inputs

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    g.load()
    A, B = inputs.gemm_inputs(w.M, w.N, w.K, w.seed)
    a, b = A.to(dev), B.to(dev)
    c = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
    tm, tn, tk = g.tile_shape(args.tile_cfg, w.M, w.N, w.K)
    tile = f"{tm}x{tn}x{tk}" + ("_pair" if tm == 256 else "")  # e.g. 256x256x128_pair
    kernel_name = "gemm_f16_f32acc_pair_kernel" if tm == 256 else "gemm_f16_f32acc_kernel"
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if args.flush_l2 else None

    def step():
        g.gemm(a, b, group_size_m=args.group_size_m, out=c, tile_cfg=args.tile_cfg)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if g.query_status(dev) != g.GEMM_OK:
        raise RuntimeError("device status after warm-up: " + g.status_string(g.GEMM_ERR_TIMEOUT))

    sampler = ClockSampler(dev.index if dev.index is not None else 0).start() if rank == 0 else None
    if sampler is not None:
        time.sleep(0.3)  # let nvidia-smi start sampling
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    n_launch0 = g.launch_count()
    t_host0 = time.time()
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    t_host1 = time.time()
    if world > 1:
        dist.barrier()
    launches = g.launch_count() - n_launch0
    status = g.query_status(dev)
    if sampler is not None:
        sampler.stop()
    per_launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    if args.flush_l2:
        total_ms = sum(per_launch_ms)
    else:
        total_ms = starts[0].elapsed_time(ends[-1])
    total_ms_max = max_over_ranks(total_ms, dev, world)

    # ---- end to end through the public API from pinned host buffers
    e2e_ms, e2e_steps, e2e_mode = run_e2e(args, w, g, A, B, dev, world)

    if rank != 0:
        return 0
    flops = 2.0 * w.M * w.N * w.K
    value = whole_job_tflops(flops, args.steps, world, total_ms_max)
    kernel_ms = statistics.fmean(per_launch_ms)
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    clocks = sampler.summary(t_host0, t_host1) if sampler is not None else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": config_dict(w, args, tile),
        "pct_of_peak": 100.0 * achieved / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak, "traffic": load_traffic(w.name, tile, args.group_size_m),
                     "peak_source": f"{peak_src} dense bf16 burst (bf16_tflops, MEASURED_PEAKS.json); "
                                    "fp16 and bf16 share the tensor rate",
                     "kernel": f"{kernel_name} {tile}", "kernel_ms": kernel_ms,
                     "flops_per_launch": flops},
        "e2e": {"value": whole_job_tflops(flops, e2e_steps, world, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": 2 * (w.M * w.K + w.K * w.N), "d2h_bytes_per_step": 2 * w.M * w.N,
                "steps": e2e_steps, "mode": e2e_mode},
        "gpu_launches": launches,
        "clocks": clocks,
        "device_status": g.status_string(status),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(A, B, w.seed, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    return 0


def run_e2e(args, w, g, A, B, dev, world):
    """Steps of host A, B -> device -> GEMM -> host C, all through the public
    API. Every step copies its own inputs in and its result out; copies of
    step i+1 and i-1 overlap the GEMM of step i (separate H2D, compute and D2H
    streams, double-buffered device operands). Returns (ms, steps, mode)."""
    import torch
    import torch.distributed as dist

    steps = max(1, min(args.steps, args.e2e_steps))
    hA, hB = A.pin_memory(), B.pin_memory()
    nbuf = 2
    dA = [torch.empty((w.M, w.K), dtype=torch.float16, device=dev) for _ in range(nbuf)]
    dB = [torch.empty((w.K, w.N), dtype=torch.float16, device=dev) for _ in range(nbuf)]
    dC = [torch.empty((w.M, w.N), dtype=torch.float16, device=dev) for _ in range(nbuf)]
    hC = [torch.empty((w.M, w.N), dtype=torch.float16).pin_memory() for _ in range(nbuf)]
    s_in, s_gemm, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    gemm_done = [None] * nbuf
    out_done = [None] * nbuf

    def step(i):
        k = i % nbuf
        with torch.cuda.stream(s_in):
            if gemm_done[k] is not None:
                s_in.wait_event(gemm_done[k])  # the GEMM that last read dA[k], dB[k]
            dA[k].copy_(hA, non_blocking=True)
            dB[k].copy_(hB, non_blocking=True)
            in_done = ev()
            in_done.record(s_in)
        with torch.cuda.stream(s_gemm):
            s_gemm.wait_event(in_done)
            if out_done[k] is not None:
                s_gemm.wait_event(out_done[k])  # the copy that last read dC[k]
            g.gemm(dA[k], dB[k], group_size_m=args.group_size_m, out=dC[k], tile_cfg=args.tile_cfg)
            gemm_done[k] = ev()
            gemm_done[k].record(s_gemm)
        with torch.cuda.stream(s_out):
            s_out.wait_event(gemm_done[k])
            hC[k].copy_(dC[k], non_blocking=True)
            out_done[k] = ev()
            out_done[k].record(s_out)

    for i in range(2):
        step(i)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_gemm.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(steps):
        step(i)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_gemm)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    return max_over_ranks(e0.elapsed_time(e1), dev, world), steps, "pipelined: H2D, GEMM and D2H streams, 2 buffers"


def main():
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="square8192")
    p.add_argument("--group-size-m", type=int, default=8)
    p.add_argument("--tile-cfg", type=int, default=0)
    p.add_argument("--flush-l2", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=50)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--reference-budget-s", type=float, default=90.0)
    args = p.parse_args()
    if args.warmup < 3:
        p.error("--warmup must be >= 3")

    from dense_fp16_gemm_fp32_gb300 import inputs
    w = inputs.WORKLOADS_BY_NAME[args.workload]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, w, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        return run_ours(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
