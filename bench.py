"""Benchmark of the bf16 -> fp32 GEMM on one GB300 (or N independent replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one tg_gemm call over the workload (4096^3 by default: the square
problem the headline TFLOP/s is quoted on), inputs already resident in HBM.
L2 is flushed between steps, outside the timed events: a 512 MB write (evicts
A, B and C) followed by a 256 MB read (evicts the flush's own dirty lines, so
their write-back does not land inside the next timed step).
Prints one JSON line (rank 0).  With --impl reference the oracle (fp64 CPU
triple loop) is timed instead, on a bounded sample of rows of the same
workload.
"""
from __future__ import annotations

import argparse
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

import synth  # noqa: E402

DEFAULT_WORKLOAD = "square_4096"
METRIC = "bf16->fp32 GEMM TFLOP/s at 1 GB300 and % of dense BF16 tensor (or HBM) roofline"
KERNEL_SOURCES = ["tiled_gemm_codegen_gb300/csrc/tg_kernel.cuh", "tiled_gemm_codegen_gb300/csrc/tg_ptx.cuh",
                  "tiled_gemm_codegen_gb300/csrc/tg_internal.h", "tiled_gemm_codegen_gb300/csrc/tg_epilogue.cuh"]
# the direct-load kernel (small problems) is its own translation unit
DIRECT_SOURCES = KERNEL_SOURCES + ["tiled_gemm_codegen_gb300/csrc/tg_direct.cu",
                                   "tiled_gemm_codegen_gb300/csrc/tg_direct.h"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal GB300 figures (dense bf16 tensor rate, HBM3e bandwidth), reported
# next to the fractions of the measured peaks.
NOMINAL_PEAKS = {"bf16_tflops": 2250.0, "hbm_gbs": 8000.0}
EXTRA_STEPS = 50  # timed steps of each non-headline workload (median reported)


# ------------------------------------------------------------------ helpers
def kernel_source_hash(direct: bool = False) -> str:
    """Hash of the sources of the kernel a plan runs: the persistent kernel,
    or (direct) the direct-load kernel."""
    import hashlib

    h = hashlib.sha256()
    for rel in (DIRECT_SOURCES if direct else KERNEL_SOURCES):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, direct: bool = False):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of the kernel the plan runs; else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    want = kernel_source_hash(direct)
    with open(TRAFFIC_FILE) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload and parts[1] == want:
                return int(parts[2])
    return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

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
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except ValueError:
                continue
            for name, val in zip(names, p[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus: int):
    """(rank, world, local_rank, torch.distributed or None)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world <= 1:
        return 0, 1, 0, None
    import torch
    import torch.distributed as dist

    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(local)
    dist.init_process_group(backend=backend)
    return rank, world, local, dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float) -> float:
    if dist is None:
        return value
    import torch

    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle timing
def oracle_sample(w, seconds: float = 10.0, max_rows: int | None = None):
    """Time the oracle (as it stands) on the first R rows of C; R is sized
    from a short calibration run to about `seconds` of CPU work."""
    import oracle

    A, B = synth.workload_inputs(w)
    a = synth.bits_u16(A if w.batch == 1 else A[0])
    b = synth.bits_u16(B if w.batch == 1 else B[0])
    threads = oracle.num_threads()
    probe = max(1, min(w.M, 32))
    t0 = time.perf_counter()
    oracle.gemm_f64(a[:probe], b, probe, w.N, w.K)
    dt = max(time.perf_counter() - t0, 1e-6)
    rows = int(max(1, min(max_rows or w.M, w.M, probe * seconds / dt)))
    t0 = time.perf_counter()
    oracle.gemm_f64(a[:rows], b, rows, w.N, w.K)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of C for one problem of {w.name} "
                      f"({rows}x{w.N}x{w.K}, {flops / 1e9:.2f} GFLOP in {dt:.2f} s)",
            "seconds": dt}


def run_reference(args, rank, world, dist):
    """--impl reference: the oracle, timed on the host cores, rank 0 only."""
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    # each step a bounded sample, so the whole run stays within a few minutes
    step_seconds = min(8.0, 150.0 / max(args.steps, 1))
    for _ in range(args.warmup and 1):
        oracle_sample(w, seconds=0.5)
    vals, secs = [], []
    last = None
    for _ in range(args.steps):
        last = oracle_sample(w, seconds=step_seconds)
        vals.append(last["value"])
        secs.append(last["seconds"])
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "batch": w.batch, "M": w.M, "N": w.N, "K": w.K,
                                        "sample": "row subset per step (bounded CPU work)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": last["cores"], "kind": "oracle",
                         "sample": last["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def roofline_of(w, ms: float, peaks: dict, peak_src: str, direct: bool = False) -> dict:
    """The binding roofline of workload `w` at `ms` per call: HBM when its
    arithmetic intensity (algorithmic flop per algorithmic byte) is below
    the ridge point of the measured peaks, else the bf16 tensor peak; the
    fraction of the nominal figure is given beside the measured one."""
    peak = float(peaks["bf16_tflops"])
    hbm = float(peaks["hbm_gbs"])
    flops = float(w.flops)
    achieved = flops / (ms * 1e-3) / 1e12
    gbs = w.bytes_moved / (ms * 1e-3) / 1e9
    if flops / w.bytes_moved < peak * 1e12 / (hbm * 1e9):
        return {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(gbs / hbm, 4), "traffic": measured_traffic(w.name, direct),
                "peak_source": f"{peak_src} hbm_gbs (copy)",
                "algorithmic_bytes_per_launch": int(w.bytes_moved),
                "nominal_peak": NOMINAL_PEAKS["hbm_gbs"],
                "nominal_frac": round(gbs / NOMINAL_PEAKS["hbm_gbs"], 4),
                "tensor_frac": round(achieved / peak, 4)}
    return {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "traffic": measured_traffic(w.name, direct),
            "peak_source": f"{peak_src} bf16_tflops (burst; kernel timed alone)",
            "algorithmic_flops_per_launch": int(flops),
            "nominal_peak": NOMINAL_PEAKS["bf16_tflops"],
            "nominal_frac": round(achieved / NOMINAL_PEAKS["bf16_tflops"], 4),
            "hbm_frac": round(gbs / hbm, 4)}


PLAN_KEYS = ("block_n", "stages", "split_k", "grid", "pack_a", "pack_b", "epilogue", "cta_pair", "stream_k",
             "sk_tiles", "direct")


def time_extra_workload(tg, torch, w, device, flush_l2, steps: int, warmup: int) -> dict:
    """One non-headline workload at its full size: `warmup` untimed calls,
    then `steps` calls each timed with CUDA events on the launching stream,
    L2 flushed before every call (outside the events)."""
    A_cpu, B_cpu = synth.workload_inputs(w)
    A, B = A_cpu.to(device), B_cpu.to(device)
    del A_cpu, B_cpu
    C = torch.empty((w.batch, w.M, w.N) if w.batch > 1 else (w.M, w.N), dtype=torch.float32, device=device)
    info = tg.plan(w.M, w.N, w.K, w.batch, A=A.data_ptr(), B=B.data_ptr(), C=C.data_ptr())
    stream = torch.cuda.current_stream(device)
    for _ in range(warmup):
        flush_l2(1.0)
        tg.gemm(A, B, C)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush_l2(float(i))
        starts[i].record(stream)
        tg.gemm(A, B, C)
        ends[i].record(stream)
    torch.cuda.synchronize()
    st = tg.device_error()
    if st != tg.TG_OK:
        raise RuntimeError(f"device error while timing {w.name}: {st}")
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    del A, B, C
    return {"per": per, "plan": {k: info[k] for k in PLAN_KEYS},
            "launches_per_step": 1 + info["pack_a"] + info["pack_b"]}


def run_gpu(args, rank, world, local, dist):
    import torch

    import tiled_gemm_codegen_gb300 as tg

    tg.load()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    w = synth.WORKLOADS[args.workload]
    f8 = args.dtype in ("e4m3", "mxfp8", "mxfp4")
    mx = args.dtype in ("mxfp8", "mxfp4")
    fp4 = args.dtype == "mxfp4"
    C = torch.empty((w.batch, w.M, w.N) if w.batch > 1 else (w.M, w.N), dtype=torch.float32, device=device)
    if fp4:
        # the same shape with packed E2M1 operands (codes drawn uniformly,
        # two a byte), A row-major and B column-major (stored N x K), E8M0
        # scales 2^-3 .. 2^3 per 32 elements of K
        lead = (w.batch,) if w.batch > 1 else ()
        A = synth.pack_fp4_codes(synth.make_fp4_codes(lead + (w.M, w.K), seed=w.seed)).to(device)
        B = synth.pack_fp4_codes(synth.make_fp4_codes(lead + (w.N, w.K), seed=w.seed + 1)).to(device)
        runs = -(-w.K // 32)
        SFA = synth.make_e8m0_codes(lead + (w.M, runs), seed=w.seed + 2).to(device)
        SFB = synth.make_e8m0_codes(lead + (w.N, runs), seed=w.seed + 3).to(device)
        launches_per_step = 2
        info = {}
    elif f8:
        # the same shape with E4M3 operands (N(0,1) draws rounded to E4M3),
        # A row-major and B column-major (stored N x K)
        lead = (w.batch,) if w.batch > 1 else ()
        A = synth.make_fp8_codes(lead + (w.M, w.K), 0, seed=w.seed, kind="normal").to(device)
        A = A.view(torch.float8_e4m3fn)
        B = synth.make_fp8_codes(lead + (w.N, w.K), 0, seed=w.seed + 1, kind="normal").to(device)
        B = B.view(torch.float8_e4m3fn)
        launches_per_step = 1
        if mx:
            # block-scaled: one E8M0 scale (2^-3 .. 2^3) per 32 elements of K;
            # the scale re-arrangement is a second launch
            runs = -(-w.K // 32)
            SFA = synth.make_e8m0_codes(lead + (w.M, runs), seed=w.seed + 2).to(device)
            SFB = synth.make_e8m0_codes(lead + (w.N, runs), seed=w.seed + 3).to(device)
            launches_per_step = 2
        info = {k: None for k in PLAN_KEYS}
    else:
        A_cpu, B_cpu = synth.workload_inputs(w)
        A = A_cpu.to(device)
        B = B_cpu.to(device)
        info = tg.plan(w.M, w.N, w.K, w.batch, A=A.data_ptr(), B=B.data_ptr(), C=C.data_ptr())
        launches_per_step = 1 + info["pack_a"] + info["pack_b"]
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    flush_read = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    sink = torch.empty((), dtype=torch.float32, device=device)

    def flush_l2(v: float):
        flush.fill_(v)                          # write > L2: A, B, C evicted
        torch.sum(flush_read, dim=0, out=sink)  # read > L2: dirty flush lines written back now

    def step():
        if fp4:
            tg.gemm_mxfp4(A, B, SFA, SFB, C)
        elif mx:
            tg.gemm_mxfp8(A, B, SFA, SFB, C)
        elif f8:
            tg.gemm_fp8(A, B, C)
        else:
            tg.gemm(A, B, C)

    # warm-up (also JIT-loads the module, allocates workspaces)
    for _ in range(args.warmup):
        flush_l2(1.0)
        step()
    torch.cuda.synchronize()
    st = tg.device_error()
    if st != tg.TG_OK:
        raise RuntimeError(f"device error during warm-up: {st}")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    # A load window right before the timed region that repeats the timed
    # steps themselves (flush, then GEMM), so that the clock samples see the
    # GPU under this benchmark's load even when the timed region itself is
    # only milliseconds long.
    t_end = time.perf_counter() + args.clock_window
    while time.perf_counter() < t_end:
        for _ in range(20):
            flush_l2(0.5)
            step()
        torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush_l2(float(i))  # outside the timed events
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    st = tg.device_error()
    if st != tg.TG_OK:
        raise RuntimeError(f"device error during timing: {st}")
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]  # ms, GEMM call only
    ms_mean = sum(per) / len(per)
    ms_max = max_over_ranks(dist, ms_mean)
    flops = float(w.flops)
    value = world * flops / (ms_max * 1e-3) / 1e12

    if f8:
        return report_f8(args, w, per, ms_mean, ms_max, world, rank, clk, wall, launches_per_step)
    # end to end through the host-buffer entry point (pinned memory)
    Ah = A_cpu.pin_memory()
    Bh = B_cpu.pin_memory()
    Ch = torch.empty(C.shape, dtype=torch.float32).pin_memory()
    tg.gemm_host(Ah, Bh, Ch)
    e2e_ms = []
    for _ in range(max(3, min(args.steps, 10))):
        flush_l2(2.0)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        tg.gemm_host(Ah, Bh, Ch)
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e_ms_max = max_over_ranks(dist, statistics.median(e2e_ms))
    e2e_value = world * flops / (e2e_ms_max * 1e-3) / 1e12

    peaks, peak_src = load_peaks()
    roofline = roofline_of(w, ms_mean, peaks, peak_src, direct=bool(info.get("direct") == 2))  # this rank's kernel

    # Every other workload at its full size, in the launch configuration of
    # the default plan: median of EXTRA_STEPS cold-L2 calls each (rank 0's
    # GPU; the replicas are identical).
    extra = {}
    extra_clk = None
    if not args.no_extra and rank == 0:
        sampler = ClockSampler(local)
        sampler.start()
        for name, wx in synth.WORKLOADS.items():
            if name == w.name:
                continue
            r = time_extra_workload(tg, torch, wx, device, flush_l2, EXTRA_STEPS, args.warmup)
            per_x = r["per"]
            med = statistics.median(per_x)
            extra[name] = {
                "batch": wx.batch, "M": wx.M, "N": wx.N, "K": wx.K, "dist": wx.dist, "seed": wx.seed,
                "steps": len(per_x), "ms_median": round(med, 4), "ms_mean": round(sum(per_x) / len(per_x), 4),
                "ms_min": round(min(per_x), 4),
                "value": round(wx.flops / (med * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "roofline": roofline_of(wx, med, peaks, peak_src, direct=r["plan"]["direct"] == 2),
                "plan": r["plan"], "gpu_launches_per_step": r["launches_per_step"],
            }
            torch.cuda.empty_cache()
        extra_clk = sampler.stop()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_sample(w, seconds=args.cpu_seconds)
        cpu.pop("seconds", None)
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "M": w.M, "N": w.N, "K": w.K,
                       "accumulate": "fp32",
                       "l2": "flushed between steps (512 MB write, then 256 MB read)",
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "plan": {k: info[k] for k in PLAN_KEYS}},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": int(A_cpu.numel() * 2 + B_cpu.numel() * 2),
                    "d2h_bytes_per_step": int(C.numel() * 4)},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": dict(clk, window=f"{args.clock_window:.1f} s of the same steps (flush, GEMM) just "
                                          "before the timed region, and the timed region"),
            "ms_min": round(min(per), 4),
            "ms_median": round(statistics.median(per), 4),
            "wall_s": round(wall, 3),
        }
        if extra:
            line["workloads"] = extra
            line["workloads_note"] = (f"each: {EXTRA_STEPS} calls after {args.warmup} warm-up calls, CUDA events "
                                      "per call, L2 flushed before every call; value and roofline from the median")
            line["workloads_clocks"] = extra_clk
        print(json.dumps(line), flush=True)


def report_f8(args, w, per, ms_mean, ms_max, world, rank, clk, wall, launches_per_step):
    """The line of an --dtype e4m3 / mxfp8 / mxfp4 run: the same shape with
    8-bit operands (mxfp8: with E8M0 block scales) or packed 4-bit ones
    (mxfp4), against the bf16 measured peak times the nominal dense
    8-bit/16-bit (2) or 4-bit/16-bit (13.5 / 2.25 = 6) tensor ratio."""
    mx = args.dtype in ("mxfp8", "mxfp4")
    fp4 = args.dtype == "mxfp4"
    peaks, peak_src = load_peaks()
    ratio = 6.0 if fp4 else 2.0
    peak = ratio * float(peaks["bf16_tflops"])
    flops = float(w.flops)
    achieved = flops / (ms_mean * 1e-3) / 1e12
    elem = 0.5 if fp4 else 1.0
    bytes_moved = w.batch * (elem * w.M * w.K + elem * w.K * w.N + 4 * w.M * w.N)
    if mx:
        bytes_moved += w.batch * (w.M + w.N) * (-(-w.K // 32))
    if rank == 0:
        line = {
            "metric": ("MXFP4 (e2m1, E8M0 scales per 32) ->fp32 GEMM TFLOP/s at 1 GB300 and % of dense FP4 "
                       "tensor roofline" if fp4 else
                       ("MXFP8 (e4m3, E8M0 scales per 32) " if mx else "e4m3") +
                       "->fp32 GEMM TFLOP/s at 1 GB300 and % of dense FP8 tensor roofline"),
            "value": round(world * flops / (ms_max * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.dtype,
            "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "M": w.M, "N": w.N, "K": w.K,
                       "layout": "A row-major, B column-major (both K-major)" +
                                 (", two E2M1 codes a byte" if fp4 else ""), "accumulate": "fp32",
                       "l2": "flushed between steps (512 MB write, then 256 MB read)"},
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4), "traffic": None,
                         "peak_source": f"{peak_src} bf16_tflops x {ratio:g} (nominal "
                                        f"{'fp4' if fp4 else 'fp8'}/bf16 dense ratio)",
                         "hbm_frac": round(bytes_moved / (ms_mean * 1e-3) / 1e9 / float(peaks["hbm_gbs"]), 4)},
            "cpu_baseline": None, "e2e": None,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": dict(clk, window=f"{args.clock_window:.1f} s of the same steps before the timed region, "
                                          "and the timed region"),
            "ms_min": round(min(per), 4), "wall_s": round(wall, 3),
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="tg", choices=["tg", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--clock-window", type=float, default=0.5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="time only the headline workload (skip the other workloads' lines)")
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "e4m3", "mxfp8", "mxfp4"],
                    help="operand type; e4m3 (mxfp8, mxfp4) runs the same shape through tg_gemm_fp8 "
                         "(tg_gemm_mxfp8, tg_gemm_mxfp4): an extra line, not the contract's metric")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "tg":
        ap.error("--warmup must be at least 3")
    rank, world, local, dist = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world, dist)
        else:
            run_gpu(args, rank, world, local, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
