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
  rate (fp16 runs at the bf16 rate) from MEASURED_PEAKS.json; traffic is the
  DRAM bytes per launch from the committed ncu summary for this kernel
  source, or null when the kernel changed since that capture.
* sustained: after the timed steps, a second timed region of back-to-back
  launches lasting at least --sustained-s seconds (default 2.5), long enough
  for the power cap to settle; its TFLOP/s, the median SM clock of the
  clock samples taken under load inside it, TFLOP/s per GHz and the fraction
  of the measured sustained bf16 rate. The timed steps of `value` are a burst
  when they last less than the power cap's settling time.
  Workloads below the ridge (fewer flops per compulsory byte than the
  measured tensor rate over the measured HBM bandwidth: the 512^3 check and
  the worked example) are judged against HBM instead: compulsory bytes
  2(MK + KN + MN) per launch over the launch time, the tensor figures beside.
* pct_of_peak: the kernel's rate against NVIDIA's published dense fp16/bf16
  tensor-core rate of one GB300 (2.25 PFLOP/s: 36 PFLOP/s per 8 GPUs with
  2:4 sparsity, halved); roofline.frac is against the measured rate.
* e2e: the same metric end to end from pinned host memory: per step the
  host-to-device copies of A and B, the GEMM, and the device-to-host copy of C.
* cpu_baseline: the CPU oracle on a bounded, seeded sample of rows of the
  same workload, timed on this host's cores (rank 0 only), plus a
  single-thread rate on a smaller sample and the host's CPU model.
* --impl reference: the oracle alone as the reference arm, on the host.
* --workload softmax_<M>x<n>: the fused row softmax instead (GB/s of 8 bytes
  per element, roofline against the measured HBM copy bandwidth).
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
# NVIDIA's published dense fp16/bf16 tensor-core rate of one GB300 (HGX B300:
# 36 PFLOP/s FP16/BF16 per 8 GPUs with 2:4 structured sparsity; dense is half)
NOMINAL_F16_TFLOPS = 2250.0
NOMINAL_F16_SOURCE = ("NVIDIA HGX B300 specification: 36 PFLOP/s FP16/BF16 tensor per 8 GPUs with 2:4 "
                      "sparsity, i.e. 2.25 PFLOP/s dense per GPU")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


KERNEL_SOURCES = {
    "gemm": ["gemm_api.cu", "gemm_kernel.cuh", "gemm_kernel_pair.cuh", "kernel_common.cuh", "ptx.cuh",
             "tile_map.cuh"],
    "softmax": ["softmax_api.cu", "softmax_kernel.cuh", "ptx.cuh"],
}


def kernel_source_hash(kind: str = "gemm") -> str:
    """Hash of the CUDA sources of one kernel family: identifies the kernel an ncu capture measured."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_fp16_gemm_fp32_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[kind]):
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


def load_traffic(key: str, kind: str = "gemm"):
    """DRAM bytes per launch recorded by ncu under `key` for this kernel source, or None."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(key)
    if not e or e.get("kernel_hash") != kernel_source_hash(kind):
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

    def idle_power(self, before: float):
        """Lowest power drawn in the samples taken before host time `before` (None if none)."""
        pw = [s[3] for s in self.samples if s[0] < before and s[3] is not None]
        return min(pw) if pw else None

    def summary(self, t0: float, t1: float, idle_w=None):
        """Clocks over the samples inside [t0, t1]. Under-load samples are those
        drawing more than a quarter of the way from the idle power (before the
        region) to the region's peak power; sm_mhz_under_load is their median."""
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed region"
        n_inside = len(inside)
        if not inside and self.samples:
            mid = 0.5 * (t0 + t1)
            inside = sorted(self.samples, key=lambda s: abs(s[0] - mid))[:3]
            window = "nearest samples (timed region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "no samples"}
        reasons = sorted({r for s in inside for r in s[4]})
        pw = [s[3] for s in inside if s[3] is not None]
        out = {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": max(s[2] for s in inside),
               "reasons": reasons, "power_w_max": max(pw) if pw else None, "samples": n_inside,
               "window": window, "seconds": t1 - t0, "period_ms": self.period_ms}
        if n_inside and pw and idle_w is not None:
            cut = idle_w + 0.25 * (max(pw) - idle_w)
            loaded = [s for s in inside if s[3] is not None and s[3] > cut]
            out["idle_w"] = idle_w
            out["samples_under_load"] = len(loaded)
            out["sm_mhz_under_load"] = statistics.median(s[1] for s in loaded) if loaded else None
        return out


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


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or "unknown"."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_rate(A, B, perm, threads: int, target_s: float):
    """(TFLOP/s, rows, seconds) of the oracle on about target_s of seeded rows."""
    import numpy as np

    M, K = A.shape
    N = B.shape[1]
    # two calibration runs separate the per-call cost (B converted to fp32 once
    # per call) from the per-row cost
    calib = min(M, max(threads, 4))
    t1 = time_oracle(A, B, np.sort(perm[:calib]), threads)
    t2 = time_oracle(A, B, np.sort(perm[:2 * calib]), threads) if 2 * calib <= M else 2 * t1
    per_row = max((t2 - t1) / calib, 1e-6)
    fixed = max(t1 - calib * per_row, 0.0)
    n = int(min(M, max(calib, (target_s - fixed) / per_row)))
    t = time_oracle(A, B, np.sort(perm[:n]), threads)
    return 2.0 * n * N * K / t / 1e12, n, t


def cpu_baseline(A, B, seed: int, target_s: float, single_s: float = 4.0):
    """The oracle as it stands on a seeded sample of rows: ~target_s of work on
    every core of this process's affinity, then ~single_s on one thread."""
    import torch
    from oracle import gemm as og

    M, K = A.shape
    N = B.shape[1]
    cores = og.default_threads()
    g = torch.Generator().manual_seed(seed + 2000)
    perm = torch.randperm(M, generator=g).numpy()
    value, n, t = oracle_rate(A, B, perm, cores, target_s)
    v1, n1, t1 = oracle_rate(A, B, perm, 1, single_s)
    return {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
            "sample": f"{n} seeded rows of the {M}x{N}x{K} workload ({n * N} outputs), "
                      f"{t:.1f} s, fp32 ascending-k C loop with {cores} threads",
            "single_thread": {"value": v1, "unit": UNIT, "cores": 1,
                              "sample": f"{n1} seeded rows of the same workload, {t1:.1f} s, one thread"}}


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
    resolved = g.tile_config(args.tile_cfg, w.M, w.N, w.K)
    tile = f"{tm}x{tn}x{tk}" + ("_pair" if tm == 256 else "")  # e.g. 256x256x128_pair
    tile += {g.TILE_256x256x64_PAIR_STREAMK: "_streamk", g.TILE_256x256x128_PAIR_ALIGNED: "_aligned",
             g.TILE_128x128x64_SPLITK: "_splitk"}.get(resolved, "")
    kernel_name = ("gemm_f16_f32acc_pair_kernel" if tm == 256 else
                   "gemm_f16_f32acc_splitk_kernel" if resolved == g.TILE_128x128x64_SPLITK else "gemm_f16_f32acc_kernel")
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if args.flush_l2 else None

    def step():
        g.gemm(a, b, group_size_m=args.group_size_m, out=c, tile_cfg=args.tile_cfg)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = g.query_status(dev)
    if st != g.GEMM_OK:
        raise RuntimeError("device status after warm-up: " + g.status_string(st))

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
    if status != g.GEMM_OK:  # a kernel gave up on a wait: the timed work is incomplete
        if sampler is not None:
            sampler.stop()
        raise RuntimeError("device status after the timed steps: " + g.status_string(status))
    per_launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    if args.flush_l2:
        total_ms = sum(per_launch_ms)
    else:
        total_ms = starts[0].elapsed_time(ends[-1])
    total_ms_max = max_over_ranks(total_ms, dev, world)

    # ---- a seconds-long region of back-to-back launches: the power-capped rate
    sustained = None
    if args.sustained_s > 0 and not args.flush_l2:
        # at most 20000 launches: below ~0.1 ms per launch the region is host-bound anyway
        n_sus = max(1, min(20000, int(args.sustained_s / max(statistics.fmean(per_launch_ms) * 1e-3, 1e-6))))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_launch1 = g.launch_count()
        t_sus0 = time.time()
        e0.record(stream)
        for _ in range(n_sus):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        t_sus1 = time.time()
        sus_launches = g.launch_count() - n_launch1
        st = g.query_status(dev)
        if st != g.GEMM_OK:
            raise RuntimeError("device status after the sustained region: " + g.status_string(st))
        sustained = {"steps": n_sus, "ms": e0.elapsed_time(e1), "launches": sus_launches,
                     "t0": t_sus0, "t1": t_sus1}

    # ---- end to end through the public API from pinned host buffers
    if sampler is not None:
        time.sleep(0.2)  # samples after the sustained region's end
        sampler.stop()
    e2e_ms, e2e_steps, e2e_mode = run_e2e(args, w, g, A, B, dev, world)

    if rank != 0:
        return 0
    flops = 2.0 * w.M * w.N * w.K
    value = whole_job_tflops(flops, args.steps, world, total_ms_max)
    kernel_ms = statistics.fmean(per_launch_ms)
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    idle_w = sampler.idle_power(t_host0) if sampler is not None else None
    clocks = sampler.summary(t_host0, t_host1, idle_w) if sampler is not None else None
    sus_line = None
    if sustained is not None:
        sus_tflops = flops * sustained["steps"] / (sustained["ms"] * 1e-3) / 1e12
        sus_clocks = sampler.summary(sustained["t0"], sustained["t1"], idle_w) if sampler is not None else None
        mhz = sus_clocks.get("sm_mhz_under_load") if sus_clocks else None
        sus_line = {"value": sus_tflops, "unit": UNIT, "seconds": sustained["ms"] * 1e-3,
                    "steps": sustained["steps"], "gpu_launches": sustained["launches"],
                    "sm_mhz_under_load": mhz,
                    "tflops_per_ghz": sus_tflops / (mhz * 1e-3) if mhz else None,
                    "peak_sustained": peak_sustained, "frac_sustained": sus_tflops / peak_sustained,
                    "peak_sustained_source": f"{peak_src} bf16 GEMM back to back for seconds under the power "
                                             "cap (bf16_tflops_sustained, MEASURED_PEAKS.json)",
                    "pct_of_nominal_peak": 100.0 * sus_tflops / NOMINAL_F16_TFLOPS,
                    "clocks": sus_clocks}
    main_s = (t_host1 - t_host0)
    # Below the ridge (peak flops / HBM bytes per second) the kernel is judged
    # against HBM: compulsory bytes 2(MK + KN + MN) per launch over its time.
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    compulsory = 2.0 * (w.M * w.K + w.K * w.N + w.M * w.N)
    ridge = peak * 1e12 / (hbm * 1e9)
    tensor_roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT, "frac": achieved / peak,
                   "traffic": load_traffic(f"{w.name}/{tile}/G{args.group_size_m}"),
                   "peak_source": f"{peak_src} dense bf16 rate of cuBLAS in a burst (bf16_tflops, "
                                  "MEASURED_PEAKS.json), the reference for a kernel timed alone; fp16 and bf16 "
                                  "share the tensor rate"}
    hbm_achieved = compulsory / (kernel_ms * 1e-3) / 1e9
    hbm_roof = {"bound": "hbm", "achieved": hbm_achieved, "peak": hbm, "unit": "GB/s", "frac": hbm_achieved / hbm,
                "traffic": tensor_roof["traffic"],
                "peak_source": f"{peak_src} HBM copy bandwidth (hbm_gbs, MEASURED_PEAKS.json)",
                "bytes_per_launch": compulsory}
    below_ridge = flops / compulsory < ridge
    roof = dict(hbm_roof if below_ridge else tensor_roof)
    roof.update({"intensity_flop_per_byte": flops / compulsory, "ridge_flop_per_byte": ridge,
                 "timed_region_s": main_s,
                 "regime": ("burst: the timed steps last less than the power cap's settling time; "
                            "the sustained key holds the power-capped rate")
                           if main_s < 1.0 else "seconds-long timed region",
                 "kernel": f"{kernel_name} {tile}", "kernel_ms": kernel_ms, "flops_per_launch": flops})
    if below_ridge:
        roof["tensor"] = {k: tensor_roof[k] for k in ("achieved", "peak", "unit", "frac")}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": config_dict(w, args, tile),
        "pct_of_peak": 100.0 * achieved / NOMINAL_F16_TFLOPS,
        "nominal_peak": {"value": NOMINAL_F16_TFLOPS, "unit": UNIT, "source": NOMINAL_F16_SOURCE},
        "roofline": roof,
        "sustained": sus_line,
        "e2e": {"value": whole_job_tflops(flops, e2e_steps, world, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": 2 * (w.M * w.K + w.K * w.N), "d2h_bytes_per_step": 2 * w.M * w.N,
                "steps": e2e_steps, "mode": e2e_mode},
        "gpu_launches": launches,
        "clocks": clocks,
        "device_status": g.status_string(status),
    }
    if not args.no_cpu_baseline and world == 1:  # the oracle's timing: one process, rank 0, N = 1
        line["cpu_baseline"] = cpu_baseline(A, B, w.seed, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    return 0


def pipelined_e2e(steps, dev, world, host_in, out_like, fn, label, nbuf=2):
    """Steps of host inputs -> device -> fn -> host output, through the public
    API. Every step copies its own inputs in and its result out; copies of
    step i+1 and i-1 overlap the compute of step i (separate H2D, compute and
    D2H streams, double-buffered device buffers). Returns (ms, steps, mode)."""
    import torch

    hin = [t.pin_memory() for t in host_in]
    din = [[torch.empty_like(t, device=dev) for t in hin] for _ in range(nbuf)]
    dout = [torch.empty_like(out_like, device=dev) for _ in range(nbuf)]
    hout = [torch.empty_like(out_like, device="cpu").pin_memory() for _ in range(nbuf)]
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    comp_done = [None] * nbuf
    out_done = [None] * nbuf

    def step(i):
        k = i % nbuf
        with torch.cuda.stream(s_in):
            if comp_done[k] is not None:
                s_in.wait_event(comp_done[k])  # the compute that last read din[k]
            for d, h in zip(din[k], hin):
                d.copy_(h, non_blocking=True)
            in_done = torch.cuda.Event()
            in_done.record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(in_done)
            if out_done[k] is not None:
                s_comp.wait_event(out_done[k])  # the copy that last read dout[k]
            fn(din[k], dout[k])
            comp_done[k] = torch.cuda.Event()
            comp_done[k].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[k])
            hout[k].copy_(dout[k], non_blocking=True)
            out_done[k] = torch.cuda.Event()
            out_done[k].record(s_out)

    for i in range(2):
        step(i)
    torch.cuda.synchronize(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_comp.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(steps):
        step(i)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_comp)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    return max_over_ranks(e0.elapsed_time(e1), dev, world), steps, f"pipelined: H2D, {label} and D2H streams, {nbuf} buffers"


def run_e2e(args, w, g, A, B, dev, world):
    import torch

    steps = max(1, min(args.steps, args.e2e_steps))
    out_like = torch.empty((w.M, w.N), dtype=torch.float16)
    return pipelined_e2e(steps, dev, world, [A, B], out_like,
                         lambda ins, out: g.gemm(ins[0], ins[1], group_size_m=args.group_size_m, out=out,
                                                 tile_cfg=args.tile_cfg), "GEMM", nbuf=args.e2e_buffers)


# ---------------------------------------------------------------- softmax workloads
SOFTMAX_METRIC = "fp32 row softmax GB/s (8 bytes per element: x read, y written)"


def softmax_config(w, args):
    mib = (4 * w.M * w.ld) >> 20
    return {"workload": w.name, "M": w.M, "n": w.n, "ld": w.ld, "seed": w.seed,
            "inputs": "x = torch.randn(fp32, host generator seeded) in rows ld wide",
            "l2": ("flush: a 256 MiB buffer is written between timed steps" if args.flush_l2 else
                   f"x and y are {mib} MiB each vs 129 MB L2" + ("" if 2 * mib > 129 else " (L2-resident)")),
            "parallelism": "replicas"}


def time_softmax_oracle(x, n, rows):
    from oracle import softmax as osm
    t = time.perf_counter()
    osm.softmax_rows(x, n, rows=rows)
    return time.perf_counter() - t


def softmax_cpu_baseline(x, w, target_s):
    """The numpy fp64 oracle on a seeded sample of rows: ~target_s of work."""
    import numpy as np
    import torch
    g = torch.Generator().manual_seed(w.seed + 2000)
    perm = torch.randperm(w.M, generator=g).numpy()
    calib = min(w.M, 64)
    per_row = max(time_softmax_oracle(x, w.n, np.sort(perm[:calib])) / calib, 1e-7)
    k = int(min(w.M, max(calib, target_s / per_row)))
    rows = np.sort(perm[:k])
    t = time_softmax_oracle(x, w.n, rows)
    return {"value": 8.0 * k * w.n / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{k} seeded rows of the {w.M}x{w.n} workload, {t:.1f} s, numpy fp64 max/exp/sum/divide"}


def run_softmax_reference(args, w, rank, world):
    if rank != 0:
        return 0
    import numpy as np
    import torch
    from dense_fp16_gemm_fp32_gb300 import inputs

    x = inputs.softmax_inputs(w.M, w.n, w.ld, w.seed).numpy()
    g = torch.Generator().manual_seed(w.seed + 3000)
    perm = torch.randperm(w.M, generator=g).numpy()
    calib = min(w.M, 64)
    per_row = max(time_softmax_oracle(x, w.n, np.sort(perm[:calib])) / calib, 1e-7)
    k = int(max(1, min(w.M, args.reference_budget_s / max(1, args.steps + args.warmup) / per_row)))
    for _ in range(args.warmup):
        time_softmax_oracle(x, w.n, np.sort(perm[:k]))
    t = 0.0
    for i in range(args.steps):
        off = (i * k) % max(1, w.M - k + 1)
        t += time_softmax_oracle(x, w.n, np.sort(perm[off:off + k]))
    value = 8.0 * k * w.n * args.steps / t / 1e9
    line = {
        "impl": "reference", "metric": SOFTMAX_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": softmax_config(w, args),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{k} seeded rows of {w.M}x{w.n} per step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_softmax(args, w, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import dense_fp16_gemm_fp32_gb300 as g
    from dense_fp16_gemm_fp32_gb300 import inputs

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    g.load()
    X = inputs.softmax_inputs(w.M, w.n, w.ld, w.seed)
    xp = X.to(dev)
    yp = torch.empty_like(xp)
    x, y = xp[:, :w.n], yp[:, :w.n]
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if args.flush_l2 else None
    plan = g.softmax_plan(w.M, w.n, dev)

    for _ in range(args.warmup):
        g.softmax(x, out=y)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index if dev.index is not None else 0).start() if rank == 0 else None
    if sampler is not None:
        time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    n_launch0 = g.softmax_launch_count()
    t_host0 = time.time()
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        starts[i].record(stream)
        g.softmax(x, out=y)
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    t_host1 = time.time()
    if world > 1:
        dist.barrier()
    launches = g.softmax_launch_count() - n_launch0
    if sampler is not None:
        sampler.stop()
    per_launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(per_launch_ms) if args.flush_l2 else starts[0].elapsed_time(ends[-1])
    total_ms_max = max_over_ranks(total_ms, dev, world)

    steps_e2e = max(1, min(args.steps, args.e2e_steps))
    e2e_ms, e2e_steps, e2e_mode = pipelined_e2e(
        steps_e2e, dev, world, [X], X, lambda ins, out: g.softmax(ins[0][:, :w.n], out=out[:, :w.n]), "softmax")

    if rank != 0:
        return 0
    nbytes = 8.0 * w.M * w.n   # algorithmic: each element read once and written once
    value = nbytes * args.steps * world / (total_ms_max * 1e-3) / 1e9
    kernel_ms = statistics.fmean(per_launch_ms)
    achieved = nbytes / (kernel_ms * 1e-3) / 1e9
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    kind = ("softmax_rows_warp_kernel" if plan["threads_per_row"] == 32 else
            "softmax_rows_cta_kernel" + (f" cluster {plan['cluster_ctas']}" if plan["cluster_ctas"] > 1 else ""))
    line = {
        "metric": SOFTMAX_METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": softmax_config(w, args),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": load_traffic(f"{w.name}/softmax", "softmax"),
                     "peak_source": f"{peak_src} HBM copy bandwidth (hbm_gbs, MEASURED_PEAKS.json)",
                     "kernel": kind, "kernel_ms": kernel_ms, "bytes_per_launch": nbytes, "plan": plan},
        "e2e": {"value": 8.0 * w.M * w.n * e2e_steps * world / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": X.numel() * 4, "d2h_bytes_per_step": X.numel() * 4,
                "steps": e2e_steps, "mode": e2e_mode},
        "gpu_launches": launches,
        "clocks": sampler.summary(t_host0, t_host1) if sampler is not None else None,
    }
    if not args.no_cpu_baseline and world == 1:  # the oracle's timing: one process, rank 0, N = 1
        line["cpu_baseline"] = softmax_cpu_baseline(X.numpy(), w, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    return 0


def main():
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="square8192")
    p.add_argument("--group-size-m", type=int, default=12,
                   help="GROUP_SIZE_M of the grouped tile order (12: the least DRAM traffic at 8192^3 with the "
                        "pair kernels' alternating k direction, measured)")
    p.add_argument("--tile-cfg", type=int, default=0)
    p.add_argument("--flush-l2", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=50)
    p.add_argument("--e2e-buffers", type=int, default=2,
                   help="device and pinned host buffer sets the end-to-end leg rotates through")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--sustained-s", type=float, default=2.5,
                   help="seconds of back-to-back launches timed after the steps (0: none)")
    p.add_argument("--reference-budget-s", type=float, default=90.0)
    args = p.parse_args()
    if args.warmup < 3:
        p.error("--warmup must be >= 3")

    from dense_fp16_gemm_fp32_gb300 import inputs
    softmax = args.workload in inputs.SOFTMAX_WORKLOADS_BY_NAME
    if softmax:
        w = inputs.SOFTMAX_WORKLOADS_BY_NAME[args.workload]
    elif args.workload in inputs.WORKLOADS_BY_NAME:
        w = inputs.WORKLOADS_BY_NAME[args.workload]
    else:
        p.error(f"unknown workload {args.workload}; one of "
                + ", ".join(list(inputs.WORKLOADS_BY_NAME) + list(inputs.SOFTMAX_WORKLOADS_BY_NAME)))

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_softmax_reference(args, w, rank, world) if softmax else run_reference(args, w, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        if softmax:
            return run_softmax(args, w, rank, world, local_rank)
        return run_ours(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
