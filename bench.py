"""Benchmark of the output-stationary tiled GEMM on GB300.

One step is one C = A @ B of the chosen workload (default: 8192^3, BF16
inputs N(0,1)/sqrt(K), FP32 accumulation, BF16 output) through the C ABI,
with A and B resident in HBM.  A + B + C take 384 MiB, more than the 129 MB
L2, so consecutive steps cannot reuse inputs from L2.  Smaller workloads
(--workload) overwrite L2 between steps, outside each step's own events.

Prints ONE JSON line (rank 0).  Keys beyond the common ones:
  roofline      dominant kernel vs the measured dense BF16 tensor peak, or vs the
                measured HBM copy bandwidth for workloads below the ridge point
  cpu_baseline  the CPU oracle on a bounded sample of the same workload
  sustained     the same step repeated for about 2.5 s after the timed region,
                with its own clock record (the power-capped rate)
  e2e           the same metric through gemm_ex_host_ws with pinned host
                buffers (host-to-device copies of A, B and the device-to-host
                copy of C inside the timed region), with the host link's
                measured GB/s and the time the copies alone allow
  clocks        SM clocks and throttle reasons sampled during the timed loop
  small_workloads  the three small named workloads: GPU time, cuBLAS time,
                and the CPU oracle on all host cores and on one thread

`--impl reference` times the CPU oracle instead (the only comparison arm:
the pages publish no implementation).  With --gpus N > 1 (under torchrun)
each rank runs an independent replica of the workload (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (1×GB300) and % of dense FP16/BF16 tensor peak, vs CPU oracle"
UNIT = "TFLOP/s"
PROFILES = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "tiled_matrix_multiplication_output_gb300", "csrc")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="square_8192_bf16")
    ap.add_argument("--kernel", default="auto")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sustained-seconds", type=float, default=2.5,
                    help="step time of the sustained leg after the timed region (0: none)")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the benchmark line: time every tensor-core variant, the "
                         "automatic choice and cuBLAS on a fixed list of BF16 shapes, one JSON "
                         "line per shape")
    ap.add_argument("--rows", action="store_true",
                    help="instead of the benchmark line: time the extended forms (transposed "
                         "operands, alpha/beta, split-K, last-wave split) on fixed BF16 "
                         "problems, one JSON line each")
    ap.add_argument("--small-sweep", action="store_true",
                    help="instead of the benchmark line: time the small-product kernels "
                         "(tile16, tc_small, tc_128x128, the SIMT kernel), the automatic choice "
                         "and cuBLAS on a fixed list of small shapes with L2 overwritten "
                         "between calls, one JSON line per shape")
    ap.add_argument("--sweep-shapes", default="",
                    help="with --small-sweep: a comma-separated list of MxNxK BF16 shapes "
                         "(BF16 output) instead of the fixed list")
    ap.add_argument("--sweep-calls", type=int, default=300,
                    help="with --small-sweep: timed calls per entry")
    ap.add_argument("--simt", action="store_true",
                    help="instead of the benchmark line: time the SIMT kernel on FP32 and "
                         "unaligned 16-bit products in every operand layout, one JSON line each")
    ap.add_argument("--kernel-only", action="store_true",
                    help="time only the GEMM launches (no e2e, cuBLAS context or CPU "
                         "baseline); used for profiler captures")
    return ap.parse_args()


# The files the benchmarked tensor-core kernel (row-major A and B) is
# compiled from; the SIMT kernel, the cost model and the other layouts are not.
KERNEL_SOURCES = ("ptx.cuh", "tc_params.h", "tc_gemm.cuh", "tc_launch.cuh", "launch.h",
                  "tc_gemm_nn.cu")


def source_digest() -> str:
    """SHA-256 over the kernel's sources: ties committed ncu counters to the
    kernel they were taken from."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def committed_traffic(kernel_name: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel
    and workload, or None if absent or taken from different sources."""
    path = os.path.join(PROFILES, f"{kernel_name}_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("source_sha256") != source_digest():
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons (every 200 ms)."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        with open(self.tmp.name) as f:
            rows = [r.strip().split(",") for r in f if r.strip()]
        os.unlink(self.tmp.name)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def dist_setup(n_gpus: int):
    import torch
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest x over all ranks (the job's time is its slowest rank's)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job TFLOP/s: every rank ran `steps` products of its own replica,
    and the job took as long as the slowest rank (max_ms)."""
    return flops_per_step * world * steps / (max_ms * 1e-3) / 1e12


def cpu_oracle_rate(A, B, target_seconds: float):
    """Time the CPU oracle on a bounded sample: the first R rows of C
    (R * N * K multiply-adds), R calibrated to about target_seconds.
    Returns (TFLOP/s, rows, seconds, threads)."""
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    N = B.shape[1]
    K = A.shape[1]
    rows = max(1, min(threads, A.shape[0]))
    t0 = time.perf_counter()
    oracle.gemm(A[:rows], B, nthreads=threads)
    dt = time.perf_counter() - t0
    rate_rows = rows / max(dt, 1e-9)
    rows = int(max(1, min(A.shape[0], rate_rows * target_seconds)))
    t0 = time.perf_counter()
    oracle.gemm(A[:rows], B, nthreads=threads)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * N * K
    return flops / dt / 1e12, rows, dt, min(threads, rows)


def reference_block(M: int, N: int, threads: int, entry_s: float, step_s: float):
    """(rows, cols) of the top-left block of C that one reference step computes.

    The oracle splits whole rows over its threads, so the block has at least
    min(threads, M) rows to keep every core busy; its width is cut to what
    one thread finishes in step_s (entry_s = one thread's time for one
    K-long entry of C), and once the full width fits, more rows are added in
    multiples of the thread count."""
    rows = max(1, min(threads, M))
    per_thread = max(1, int(step_s / max(entry_s, 1e-12)))
    if per_thread < N:
        return rows, per_thread
    rounds = max(1, per_thread // N)
    return max(1, min(M, rows * rounds)), N


def run_reference(args, rank, world):
    """The CPU oracle as the comparison arm: each step is a bounded sample
    (the top-left rows x cols block of C, full K) of the same workload."""
    from tiled_matrix_multiplication_output_gb300 import inputs
    import oracle
    if rank != 0:
        return
    w = inputs.WORKLOADS[args.workload]
    A, B = inputs.make(w)
    oracle.build()
    threads = os.cpu_count() or 1
    # calibrate: one thread's time per entry of C, from one probe row each
    probe_rows = max(1, min(threads, w.M))
    probe_cols = max(1, min(w.N, 512))
    Bp = B[:, :probe_cols].contiguous()
    t0 = time.perf_counter()
    oracle.gemm(A[:probe_rows], Bp, nthreads=threads)
    entry_s = (time.perf_counter() - t0) / probe_cols
    # warmup + steps take about two minutes
    step_s = 120.0 / max(1, args.steps + args.warmup)
    rows, cols = reference_block(w.M, w.N, threads, entry_s, step_s)
    As, Bs = A[:rows].contiguous(), B[:, :cols].contiguous()
    for _ in range(args.warmup):
        oracle.gemm(As, Bs, nthreads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemm(As, Bs, nthreads=threads)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * cols * w.K * args.steps
    value = flops / dt / 1e12
    sample = (f"top-left {rows}x{cols} block of the {w.M}x{w.N} C per step "
              f"({rows}x{cols}x{w.K}), FP64 i-k-j loop over the rounded inputs")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, "cpu_oracle"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(threads, rows),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


L2_BYTES = 129e6   # GB300 L2 capacity
ALU_SMS = 152      # GB300 SMs, for the FP32 FMA peak
# Dense FP16/BF16 tensor rate of one SM: a cta_group::1 tcgen05.mma of
# M=128, N=256, K=16 (524,288 multiply-adds) takes 128 cycles, i.e. 4096
# multiply-adds = 8192 FLOP per cycle per SM.
TENSOR_FLOP_PER_SM_CYCLE = 8192


def theoretical_tensor_tflops(sms: int, mhz: float) -> float:
    """Dense FP16/BF16 tensor peak: SMs x 8192 FLOP per cycle x clock."""
    return sms * TENSOR_FLOP_PER_SM_CYCLE * mhz * 1e6 / 1e12


def footprint_bytes(w):
    in_b = 4 if w.in_dtype == "f32" else 2
    out_b = 4 if w.out_dtype == "f32" else 2
    return (w.M * w.K + w.K * w.N) * in_b + w.M * w.N * out_b


def needs_flush(w) -> bool:
    """Whether A, B and C together fit in L2, so that consecutive steps would
    find their inputs there: such workloads flush L2 between steps."""
    return footprint_bytes(w) <= L2_BYTES


def roofline_of(w, flops, avg_launch_ms, peaks, peak_kind, traffic, sms=ALU_SMS, run_mhz=None):
    """The roofline object for one workload.  The bound follows from the
    arithmetic intensity (FLOPs per compulsory byte of A, B and C) against
    the ridge point of the compute peak over the HBM peak: below it the
    workload is HBM-bound (achieved = compulsory bytes / time, against the
    measured copy bandwidth), above it compute-bound -- the tensor cores for
    16-bit inputs (measured cuBLAS BF16 peak), the FP32 FMA pipes for FP32
    inputs (peak derived: SMs x 128 lanes x 2 FLOP x the maximum SM clock).
    A tensor-bound line also carries the theoretical dense peak (SMs x 8192
    FLOP per cycle x the maximum SM clock, and x the clock sampled during
    the run when run_mhz is given) and the fractions of both."""
    seconds = avg_launch_ms * 1e-3
    nbytes = footprint_bytes(w)
    hbm = float(peaks["hbm_gbs"])
    if w.in_dtype == "f32":
        compute, kind = ALU_SMS * 128 * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12, "alu"
        source = f"derived: {ALU_SMS} SMs x 128 FP32 lanes x 2 FLOP x the maximum SM clock"
    else:
        compute, kind = float(peaks["bf16_tflops"]), "tensor"
        source = f"{peak_kind} bf16_tflops (burst)"
    timing = ("CUDA events around every step on the launching stream; a step is the main "
              "kernel plus, when tiles are split, the small reduction, so the main kernel's "
              "share is slightly understated")
    if flops / nbytes < compute * 1e12 / (hbm * 1e9):
        achieved = nbytes / seconds / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": traffic, "timing": timing,
                "algorithmic_bytes": nbytes, "peak_source": f"{peak_kind} hbm_gbs"}
    achieved = flops / seconds / 1e12
    line = {"bound": kind, "achieved": achieved, "peak": compute, "unit": UNIT,
            "frac": achieved / compute, "traffic": traffic, "timing": timing,
            "peak_source": source}
    if kind == "tensor":
        line["frac_of_sustained"] = achieved / float(peaks["bf16_tflops_sustained"])
        max_mhz = float(peaks.get("sm_max_mhz", 2070.0))
        theo = theoretical_tensor_tflops(sms, max_mhz)
        line["theoretical_peak"] = theo
        line["frac_of_theoretical"] = achieved / theo
        line["theoretical_source"] = (f"{sms} SMs x {TENSOR_FLOP_PER_SM_CYCLE} dense FP16/BF16 "
                                      f"FLOP per cycle (one 128x256x16 tcgen05.mma per 128 "
                                      f"cycles) x {max_mhz:.0f} MHz maximum SM clock")
        if run_mhz:
            at_run = theoretical_tensor_tflops(sms, float(run_mhz))
            line["theoretical_peak_at_run_clock"] = at_run
            line["frac_of_theoretical_at_run_clock"] = achieved / at_run
            line["run_clock_mhz"] = float(run_mhz)
    return line


def config_of(w, kernel):
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "in_dtype": w.in_dtype,
            "acc_dtype": "f32", "out_dtype": w.out_dtype, "layout": "row-major A, B, C",
            "kernel": kernel, "dist": w.dist, "seed": w.seed,
            "l2": ("L2 flushed between steps (a 2 x L2 write outside each step's events); "
                   "time = sum of per-step event times") if needs_flush(w)
            else "A+B+C larger than L2"}


def timed_loop(fn, steps, stream, flush_buf):
    """Runs fn `steps` times on `stream` and returns (total_ms, per-step ms).
    Without a flush buffer the steps run back to back between two events
    (per-step events in between); with one, every step has its own pair of
    events and L2 is overwritten between steps, outside them."""
    import torch
    if flush_buf is None:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        ev[0].record(stream)
        for i in range(steps):
            fn()
            ev[i + 1].record(stream)
        torch.cuda.synchronize(stream.device)
        per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
        return ev[0].elapsed_time(ev[-1]), per
    es = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        es[i].record(stream)
        fn()
        ee[i].record(stream)
        flush_buf.zero_()
    torch.cuda.synchronize(stream.device)
    per = [es[i].elapsed_time(ee[i]) for i in range(steps)]
    return sum(per), per


def sustained_leg(fn, ms_per_step, stream, flush_buf, gpu_index, seconds=2.5, max_steps=20000):
    """Back-to-back steps for about `seconds` of step time after the timed
    region, with their own clock record: the rate once the power cap has
    settled, where the timed region may be a short burst."""
    steps = int(max(10, min(max_steps, math.ceil(seconds * 1e3 / max(ms_per_step, 1e-4)))))
    sampler = ClockSampler(gpu_index)
    sampler.start()
    time.sleep(0.25)
    total_ms, _ = timed_loop(fn, steps, stream, flush_buf)
    clocks = sampler.stop()
    return steps, total_ms, clocks


def link_rates(host_in, dev_in, dev_out, host_out, stream, reps=5):
    """Host link GB/s from pinned buffers: host-to-device copies of the
    inputs alone, the device-to-host copy of the output alone, and both at
    once on two streams (median of `reps`, CUDA events)."""
    import torch
    side = torch.cuda.Stream(device=stream.device)
    h2d_bytes = sum(t.numel() * t.element_size() for t in host_in)
    d2h_bytes = host_out.numel() * host_out.element_size()

    def timed(kind):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(stream.device)
        e0.record(stream)
        side.wait_event(e0)
        if kind in ("h2d", "both"):
            with torch.cuda.stream(stream):
                for d, h in zip(dev_in, host_in):
                    d.copy_(h, non_blocking=True)
        if kind in ("d2h", "both"):
            with torch.cuda.stream(side if kind == "both" else stream):
                host_out.copy_(dev_out, non_blocking=True)
        if kind == "both":
            stream.wait_stream(side)
        e1.record(stream)
        torch.cuda.synchronize(stream.device)
        return e0.elapsed_time(e1)

    out = {}
    for kind, nbytes in (("h2d", h2d_bytes), ("d2h", d2h_bytes), ("both", h2d_bytes + d2h_bytes)):
        timed(kind)
        ms = statistics.median(timed(kind) for _ in range(reps))
        out[f"{kind}_gbs"] = nbytes / (ms * 1e-3) / 1e9
        out[f"{kind}_ms"] = ms
    return out


SMALL_WORKLOADS = ("worked_9x9", "square_128_f16", "edge_96x200x1000_bf16")


def trimmed_mean(xs, cut=0.1):
    """Mean of the middle (1 - 2 cut) of the values: event times of a few
    microseconds come in steps of about half a microsecond, so a median
    jumps between steps where a trimmed mean does not."""
    v = sorted(xs)
    k = int(len(v) * cut)
    v = v[k:len(v) - k] or v
    return sum(v) / len(v)


def oracle_seconds(A, B, threads, min_seconds=0.2, min_reps=3):
    """Median wall time of one full oracle product on `threads` threads."""
    import oracle
    times = []
    t_end = time.perf_counter() + min_seconds
    while len(times) < min_reps or time.perf_counter() < t_end:
        t0 = time.perf_counter()
        oracle.gemm(A, B, nthreads=threads)
        times.append(time.perf_counter() - t0)
        if len(times) >= 1000:
            break
    return statistics.median(times)


def small_workload_lines(dev, flush_buf_bytes):
    """For each small named workload: the GPU time of the benchmarked call
    (gemm_ex_ws, automatic choice; median and trimmed mean of 400 steps with
    L2 overwritten between them), cuBLAS on the same 16-bit inputs, and the
    full CPU oracle product on all host cores and on one thread."""
    import torch
    import oracle
    import tiled_matrix_multiplication_output_gb300 as tg
    from tiled_matrix_multiplication_output_gb300 import binding, inputs
    oracle.build()
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(int(flush_buf_bytes), dtype=torch.uint8, device=dev)
    threads = os.cpu_count() or 1
    lines = []
    for name in SMALL_WORKLOADS:
        w = inputs.WORKLOADS[name]
        A_cpu, B_cpu = inputs.make(w)
        A, B = A_cpu.to(dev), B_cpu.to(dev)
        C = torch.empty((w.M, w.N), dtype=binding.torch_dtype(w.out_dtype), device=dev)
        ws_bytes = max(16, tg.gemm_workspace_size(w.M, w.N, w.K))
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        in_code, out_code = binding.dtype_code(w.in_dtype), binding.dtype_code(w.out_dtype)

        def step():
            rc = tg.gemm_ex_ws(A.data_ptr(), B.data_ptr(), C.data_ptr(), w.M, w.N, w.K, in_code,
                               tg.F32, out_code, ws.data_ptr(), ws_bytes, stream.cuda_stream)
            if rc != 0:
                raise tg.GemmError(rc, "gemm_ex_ws")

        for _ in range(5):
            step()
        _, per = timed_loop(step, 400, stream, flush)
        gpu_us = statistics.median(per) * 1e3
        gpu_us_mean = trimmed_mean(per) * 1e3
        chosen = tg.gemm_select_kernel(A.data_ptr(), B.data_ptr(), C.data_ptr(), w.M, w.N, w.K,
                                       in_code, tg.F32, out_code)
        line = {"workload": name, "M": w.M, "N": w.N, "K": w.K, "in_dtype": w.in_dtype,
                "out_dtype": w.out_dtype, "kernel": tg.KERNEL_NAMES.get(chosen, str(chosen)),
                "gpu_us": gpu_us, "gpu_us_trimmed_mean": gpu_us_mean,
                "gpu_tflops": w.flops / (gpu_us * 1e-6) / 1e12,
                "gpu_gbs_compulsory": footprint_bytes(w) / (gpu_us * 1e-6) / 1e9}
        if w.in_dtype != "f32":
            for _ in range(5):
                torch.matmul(A, B)
            _, per = timed_loop(lambda: torch.matmul(A, B), 400, stream, flush)
            line["cublas_us"] = statistics.median(per) * 1e3
            line["cublas_us_trimmed_mean"] = trimmed_mean(per) * 1e3
        cpu = {}
        for label, nthr in (("all_cores", threads), ("one_thread", 1)):
            sec = oracle_seconds(A_cpu, B_cpu, nthr)
            cpu[label] = {"value": w.flops / sec / 1e12, "unit": UNIT, "us": sec * 1e6,
                          "cores": min(nthr, w.M)}
        line["cpu_baseline"] = {"kind": "oracle", "sample": "the whole product", **cpu}
        lines.append(line)
        del A, B, C, ws
    del flush
    return lines


def run_ours(args, rank, world, local):
    import torch
    import tiled_matrix_multiplication_output_gb300 as tg
    from tiled_matrix_multiplication_output_gb300 import binding, inputs

    tg.load_library(build_if_missing=True)
    w = inputs.WORKLOADS[args.workload]
    A_cpu, B_cpu = inputs.make(w)
    dev = torch.device("cuda", local)
    A = A_cpu.to(dev)
    B = B_cpu.to(dev)
    odt = binding.torch_dtype(w.out_dtype)
    C = torch.empty((w.M, w.N), dtype=odt, device=dev)
    in_code = binding.dtype_code(w.in_dtype)
    out_code = binding.dtype_code(w.out_dtype)
    kid = tg.KERNELS[args.kernel]
    chosen = kid if kid != 0 else tg.gemm_select_kernel(
        A.data_ptr(), B.data_ptr(), C.data_ptr(), w.M, w.N, w.K, in_code, tg.F32, out_code)
    kname = tg.KERNEL_NAMES.get(chosen, str(chosen))
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    # The automatic path goes through gemm_ex_ws with a workspace allocated
    # here, before any timing: on the CTA-pair kernel it splits the tiles of
    # the last, partial wave along K, and products with few tiles and a long
    # K are split along K throughout (a second, small launch sums the pieces).
    use_ws = kid == 0
    ws_bytes = tg.gemm_workspace_size(w.M, w.N, w.K) if use_ws else 0
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    ws_splits = tg.gemm_ws_split_count(w.M, w.N, w.K, in_code, tg.F32, out_code) if use_ws else 0
    if ws_splits > 0:
        kname = f"tc_128x128+split_k{ws_splits}"
    elif use_ws and chosen == tg.KERNELS["tc_256x256"]:
        kname = "tc_256x256+split_last_wave"

    def step():
        if use_ws:
            rc = tg.gemm_ex_ws(A.data_ptr(), B.data_ptr(), C.data_ptr(), w.M, w.N, w.K, in_code,
                               tg.F32, out_code, ws.data_ptr(), ws_bytes, sh)
        else:
            rc = tg.gemm_ex_kernel(A.data_ptr(), B.data_ptr(), C.data_ptr(), w.M, w.N, w.K,
                                   in_code, tg.F32, out_code, chosen, sh)
        if rc != 0:
            raise tg.GemmError(rc, "gemm_ex_ws" if use_ws else "gemm_ex_kernel")

    for _ in range(args.warmup if args.kernel_only else max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    rc = tg.gemm_device_status(sh)
    if rc != 0:
        raise tg.GemmError(rc, "warm-up")

    # ---- timed region: K steps, events around every launch
    flush_buf = (torch.empty(int(2 * L2_BYTES), dtype=torch.uint8, device=dev)
                 if needs_flush(w) else None)
    sampler = ClockSampler(local) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.start()
        time.sleep(0.25)
    launches0 = tg.gemm_launch_count()
    total_ms, per_launch = timed_loop(step, args.steps, stream, flush_buf)
    launches = tg.gemm_launch_count() - launches0
    barrier(world)
    clocks = sampler.stop() if sampler else None
    rc = tg.gemm_device_status(sh)
    if rc != 0:
        raise tg.GemmError(rc, "timed region")
    total_ms = max_over_ranks(total_ms, world)
    ms_per_step = total_ms / args.steps
    flops = float(w.flops)
    value = job_rate(flops, args.steps, world, total_ms)

    if args.kernel_only:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                              "steps": args.steps, "warmup": args.warmup,
                              "ms_per_step": ms_per_step, "config": config_of(w, kname),
                              "gpu_launches": launches, "kernel_only": True}), flush=True)
        return

    # ---- the same step held for seconds: the power-capped rate
    sustained = None
    if args.sustained_seconds > 0:
        sus_steps, sus_ms, sus_clocks = sustained_leg(step, ms_per_step, stream, flush_buf, local,
                                                      seconds=args.sustained_seconds)
        sus_ms = max_over_ranks(sus_ms, world)
        sustained = {"value": job_rate(flops, sus_steps, world, sus_ms), "unit": UNIT,
                     "steps": sus_steps, "ms_per_step": sus_ms / sus_steps,
                     "seconds": sus_ms * 1e-3, "clocks": sus_clocks}

    # ---- end to end through the host-buffer entry point
    in_b = 4 if w.in_dtype == "f32" else 2
    out_b = 4 if w.out_dtype == "f32" else 2
    Ah = A_cpu.pin_memory()
    Bh = B_cpu.pin_memory()
    Ch = torch.empty((w.M, w.N), dtype=odt).pin_memory()
    e2e_steps = max(1, min(args.e2e_steps, args.steps))

    def host_step():
        rc = tg.gemm_ex_host_ws(Ah.data_ptr(), Bh.data_ptr(), Ch.data_ptr(), w.M, w.N, w.K,
                                in_code, tg.F32, out_code, A.data_ptr(), B.data_ptr(),
                                C.data_ptr(), ws.data_ptr(), ws_bytes if use_ws else 0, sh)
        if rc != 0:
            raise tg.GemmError(rc, "gemm_ex_host_ws")

    for _ in range(3):
        host_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        host_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / e2e_steps
    e2e_value = flops * world / (e2e_ms * 1e-3) / 1e12
    h2d_bytes = (w.M * w.K + w.K * w.N) * in_b
    d2h_bytes = w.M * w.N * out_b
    link = link_rates((Ah, Bh), (A, B), C, Ch, stream)
    panel_rows = tg.gemm_host_panel_rows(w.M)
    panels = max(1, -(-w.M // max(1, panel_rows)))
    # what the copies alone allow: every byte over the link with both
    # directions busy, plus the one panel's product that cannot overlap a copy
    model_ms = (h2d_bytes + d2h_bytes) / (link["both_gbs"] * 1e9) * 1e3 + ms_per_step / panels
    link.update({"panels": panels, "panel_rows": panel_rows, "model_ms": model_ms, "e2e_over_model": e2e_ms / model_ms,
                 "achieved_gbs": (h2d_bytes + d2h_bytes) / (e2e_ms * 1e-3) / 1e9})

    # ---- cuBLAS on the same inputs, as context only
    for _ in range(5):
        torch.matmul(A, B)
    n_cublas = args.steps   # same length as our timed loop
    cublas_ms, _ = timed_loop(lambda: torch.matmul(A, B), n_cublas, stream, flush_buf)
    cublas_tflops = flops * n_cublas / (cublas_ms * 1e-3) / 1e12
    cublas_sustained, cb_clocks = None, None
    if args.sustained_seconds > 0:
        cb_steps, cb_ms, cb_clocks = sustained_leg(lambda: torch.matmul(A, B), cublas_ms / n_cublas,
                                                   stream, flush_buf, local,
                                                   seconds=args.sustained_seconds)
        cublas_sustained = flops * cb_steps / (cb_ms * 1e-3) / 1e12

    if rank != 0:
        return
    peaks, peak_kind = load_peaks()
    avg_launch_ms = statistics.mean(per_launch)
    base_kernel = kname.split("+")[0]
    traffic = committed_traffic(
        f"tc_gemm_{base_kernel[3:]}" if base_kernel.startswith("tc_") else base_kernel, w.name)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    roofline = roofline_of(w, flops, avg_launch_ms, peaks, peak_kind, traffic, sms=sms,
                           run_mhz=(clocks or {}).get("sm_mhz"))
    if roofline["bound"] == "tensor" and sustained:
        sustained["frac_of_sustained_peak"] = sustained["value"] / float(
            peaks["bf16_tflops_sustained"])
        if sustained["clocks"] and sustained["clocks"].get("sm_mhz"):
            sustained["frac_of_theoretical_at_run_clock"] = sustained["value"] / (
                theoretical_tensor_tflops(sms, sustained["clocks"]["sm_mhz"]) * world)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.in_dtype, "data": "synthetic",
        "config": config_of(w, kname),
        "roofline": roofline,
        "sustained": sustained,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d_bytes,
                "d2h_bytes_per_step": d2h_bytes, "steps": e2e_steps, "ms_per_step": e2e_ms,
                "entry_point": "gemm_ex_host_ws (pinned host buffers, the same workspace)",
                "link": link},
        "gpu_launches": launches,
        "clocks": clocks,
        "context": {"cublas_torch_matmul_tflops": cublas_tflops,
                    "cublas_sustained_tflops": cublas_sustained, "cublas_sustained_clocks": cb_clocks,
                    "per_launch_ms_min": min(per_launch), "per_launch_ms_median":
                    statistics.median(per_launch)},
    }
    if world == 1 and not args.no_cpu_baseline:
        v, rows, secs, cores = cpu_oracle_rate(A_cpu, B_cpu, args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"first {rows} of {w.M} rows of C ({rows}x{w.N}x{w.K}), {secs:.1f} s"}
        if w.name not in SMALL_WORKLOADS:
            line["small_workloads"] = small_workload_lines(dev, 2 * L2_BYTES)
    print(json.dumps(line), flush=True)


SWEEP_SHAPES = [(n, n, n) for n in (2048, 3072, 4096, 6144, 8192)] + [
    (256, 8192, 4096), (8192, 256, 4096), (1024, 4096, 8192), (2048, 2048, 16384),
    (12288, 12288, 2048), (1536, 1536, 1536), (2560, 2560, 2560), (5120, 5120, 1024)]


def median_call_ms(f, steps):
    """Median CUDA-event time in ms of one call of f, after 5 untimed calls."""
    import torch
    for _ in range(5):
        f()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record()
    for i in range(steps):
        f()
        ev[i + 1].record()
    torch.cuda.synchronize()
    return statistics.median([ev[i].elapsed_time(ev[i + 1]) for i in range(steps)])


def run_sweep():
    """Median per-call TFLOP/s of each tensor-core variant, the automatic
    choice and cuBLAS (torch.matmul) on BF16 inputs, BF16 output."""
    import torch
    import tiled_matrix_multiplication_output_gb300 as tg
    tg.load_library(build_if_missing=True)
    torch.cuda.set_device(0)

    timeit = median_call_ms

    g = torch.Generator(device="cuda").manual_seed(0)
    for M, N, K in SWEEP_SHAPES:
        A = (torch.randn(M, K, device="cuda", generator=g) / math.sqrt(K)).bfloat16()
        B = (torch.randn(K, N, device="cuda", generator=g) / math.sqrt(K)).bfloat16()
        C = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
        steps = max(20, min(300, int(2e12 / (2 * M * N * K))))
        flops = 2.0 * M * N * K
        row = {"shape": [M, N, K]}
        for k in ("tc_128x128", "tc_128x256", "tc_256x256", "tc_256x128", "auto"):
            ms = timeit(lambda: tg.matmul(A, B, out_dtype=torch.bfloat16, out=C, kernel=k), steps)
            row[k] = round(flops / ms / 1e9, 1)
        row["auto_pick"] = tg.KERNEL_NAMES[tg.gemm_select_kernel(
            A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, tg.BF16, tg.F32, tg.BF16)]
        row["cublas"] = round(flops / timeit(lambda: torch.matmul(A, B), steps) / 1e9, 1)
        print(json.dumps(row), flush=True)


SMALL_SWEEP_SHAPES = [
    ("bf16", "bf16", 64, 64, 64), ("bf16", "bf16", 128, 128, 128), ("bf16", "bf16", 96, 200, 1000),
    ("bf16", "bf16", 128, 128, 1024), ("bf16", "bf16", 192, 192, 192), ("bf16", "bf16", 256, 256, 256),
    ("bf16", "bf16", 256, 128, 512), ("bf16", "bf16", 64, 64, 2048), ("bf16", "bf16", 128, 128, 2048),
    ("bf16", "bf16", 32, 1024, 256), ("bf16", "bf16", 256, 256, 512), ("bf16", "bf16", 384, 384, 128),
    ("bf16", "bf16", 512, 512, 128), ("bf16", "bf16", 128, 128, 512), ("bf16", "bf16", 160, 160, 640),
    ("bf16", "bf16", 256, 256, 1024), ("bf16", "bf16", 192, 192, 1024), ("bf16", "bf16", 320, 320, 256),
    ("bf16", "bf16", 384, 384, 384), ("bf16", "bf16", 512, 512, 512), ("bf16", "bf16", 64, 1024, 1024),
    ("f16", "f32", 128, 128, 128), ("bf16", "f32", 96, 200, 1000),
    ("f32", "f32", 128, 128, 128), ("f32", "f32", 100, 200, 1000), ("f32", "f32", 512, 512, 512),
    ("f32", "f32", 640, 640, 640), ("f32", "f32", 768, 768, 768)]


def parse_sweep_shapes(arg):
    """'MxNxK,MxNxK,...' -> [("bf16", "bf16", M, N, K), ...]; empty -> the
    fixed list.  Sizes must be positive integers."""
    if not arg:
        return list(SMALL_SWEEP_SHAPES)
    shapes = []
    for item in arg.split(","):
        dims = item.strip().lower().split("x")
        if len(dims) != 3 or not all(d.isdigit() and int(d) > 0 for d in dims):
            raise ValueError(f"bad shape {item!r}: want MxNxK with positive sizes")
        shapes.append(("bf16", "bf16") + tuple(int(d) for d in dims))
    return shapes


def run_small_sweep(shapes_arg="", calls=300):
    """Per-call GPU time (microseconds, trimmed mean of `calls` calls with L2
    overwritten between them, outside the events) of each small-product
    kernel forced, of the automatic choice through gemm_ex_ws, and of
    cuBLAS (torch.matmul, TF32 off) on N(0, 1) inputs."""
    import torch
    import tiled_matrix_multiplication_output_gb300 as tg
    tg.load_library(build_if_missing=True)
    torch.cuda.set_device(0)
    torch.backends.cuda.matmul.allow_tf32 = False
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(int(2 * L2_BYTES), dtype=torch.uint8, device=dev)
    dt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
    g = torch.Generator(device="cuda").manual_seed(0)

    def us(fn):
        for _ in range(min(5, calls)):
            fn()
        _, per = timed_loop(fn, max(1, calls), stream, flush)
        return round(trimmed_mean(per) * 1e3, 2)

    for in_dt, out_dt, M, N, K in parse_sweep_shapes(shapes_arg):
        A = torch.randn(M, K, device=dev, generator=g).to(dt[in_dt])
        B = torch.randn(K, N, device=dev, generator=g).to(dt[in_dt])
        C = torch.empty(M, N, device=dev, dtype=dt[out_dt])
        ic, oc = tg.binding.dtype_code(dt[in_dt]), tg.binding.dtype_code(dt[out_dt])
        row = {"shape": [M, N, K], "in": in_dt, "out": out_dt}
        kernels = ("tile16", "simt") if in_dt == "f32" else ("tile16", "tc_small", "tc_128x128", "simt")
        for k in kernels:
            kid = tg.KERNELS[k]
            row[k] = us(lambda: tg.gemm_ex_kernel(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                                  ic, tg.F32, oc, kid, stream.cuda_stream))
        ws_bytes = max(16, tg.gemm_workspace_size(M, N, K))
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        row["auto"] = us(lambda: tg.gemm_ex_ws(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, ic,
                                               tg.F32, oc, ws.data_ptr(), ws_bytes,
                                               stream.cuda_stream))
        row["auto_pick"] = tg.KERNEL_NAMES[tg.gemm_select_kernel(
            A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, ic, tg.F32, oc)]
        row["cublas"] = us(lambda: torch.matmul(A, B))
        rc = tg.gemm_device_status(stream.cuda_stream)
        if rc != 0:
            raise tg.GemmError(rc, "small sweep")
        print(json.dumps(row), flush=True)


SIMT_SHAPES = [("f32", 4096, 4096, 4096), ("f32", 8192, 8192, 1024), ("f32", 2048, 2048, 2048),
               ("bf16", 4095, 4095, 4095)]


def run_simt():
    """Median per-call TFLOP/s of the SIMT kernel (forced) on FP32 inputs and
    on 16-bit inputs whose odd row pitch keeps them off the tensor cores, in
    every operand layout, FP32 output; cuBLAS FP32 (TF32 off) beside the
    row-major FP32 products, and the FP32 FMA peak at the maximum SM clock
    (152 SMs x 128 lanes x 2 FLOP x 2.07 GHz) for scale.  A last line gives
    the SM clocks sampled over the run."""
    import torch
    import tiled_matrix_multiplication_output_gb300 as tg
    tg.load_library(build_if_missing=True)
    torch.cuda.set_device(0)
    torch.backends.cuda.matmul.allow_tf32 = False
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    fma_peak = sms * 128 * 2 * 2.07e9 / 1e12
    dt = {"f32": torch.float32, "bf16": torch.bfloat16}
    g = torch.Generator(device="cuda").manual_seed(0)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    for name, M, N, K in SIMT_SHAPES:
        flops = 2.0 * M * N * K
        steps = max(10, min(100, int(2e11 / flops)))
        for op_a, op_b in (("n", "n"), ("t", "n"), ("n", "t"), ("t", "t")):
            A = torch.randn((K, M) if op_a == "t" else (M, K), device="cuda", generator=g).to(dt[name])
            B = torch.randn((N, K) if op_b == "t" else (K, N), device="cuda", generator=g).to(dt[name])
            C = torch.empty((M, N), device="cuda", dtype=torch.float32)
            ms = median_call_ms(lambda: tg.addmm(A, B, C, op_a=op_a, op_b=op_b, kernel="simt"),
                                steps)
            row = {"in_dtype": name, "shape": [M, N, K], "layout": op_a + op_b,
                   "us": round(ms * 1e3, 1), "tflops": round(flops / ms / 1e9, 2),
                   "fma_peak_tflops_at_max_clock": round(fma_peak, 1)}
            if name == "f32" and op_a == "n" and op_b == "n":
                cb = median_call_ms(lambda: torch.matmul(A, B, out=C), steps)
                row["cublas_f32_tflops"] = round(flops / cb / 1e9, 2)
            print(json.dumps(row), flush=True)
            del A, B, C
    print(json.dumps({"clocks": clocks.stop()}), flush=True)


def run_rows():
    """Median per-call time and TFLOP/s of the extended entry points."""
    import torch
    import tiled_matrix_multiplication_output_gb300 as tg
    tg.load_library(build_if_missing=True)
    torch.cuda.set_device(0)

    timeit = median_call_ms

    def emit(row, M, N, K, ms, **extra):
        print(json.dumps({"row": row, "shape": [M, N, K], "us": round(ms * 1e3, 2),
                          "tflops": round(2.0 * M * N * K / ms / 1e9, 1), **extra}), flush=True)

    g = torch.Generator(device="cuda").manual_seed(0)
    n = 8192
    A0 = (torch.randn(n, n, device="cuda", generator=g) / math.sqrt(n)).bfloat16()
    B0 = (torch.randn(n, n, device="cuda", generator=g) / math.sqrt(n)).bfloat16()
    C = torch.empty(n, n, device="cuda", dtype=torch.bfloat16)
    # f1: operand layouts on the pair kernel
    for op_a, op_b in (("n", "n"), ("t", "n"), ("n", "t"), ("t", "t")):
        A = A0.t().contiguous() if op_a == "t" else A0
        B = B0.t().contiguous() if op_b == "t" else B0
        ms = timeit(lambda: tg.addmm(A, B, C, op_a=op_a, op_b=op_b), 200)
        emit("f1_layout_" + op_a + op_b, n, n, n, ms)
    # f2: accumulate into C (reads C: 128 MiB more traffic per call)
    ms = timeit(lambda: tg.addmm(A0, B0, C, alpha=1.0, beta=1.0), 200)
    emit("f2_addmm_beta1", n, n, n, ms)
    ms = timeit(lambda: tg.addmm(A0, B0, C, alpha=0.5, beta=0.0), 200)
    emit("f2_alpha_only", n, n, n, ms)
    del A0, B0, C
    # f4: split-K on few-tile, long-K products; last-wave split on squares
    for M, N, K in ((96, 200, 1000), (256, 256, 16384), (512, 512, 65536), (128, 1024, 8192)):
        A = (torch.randn(M, K, device="cuda", generator=g) / math.sqrt(K)).bfloat16()
        B = (torch.randn(K, N, device="cuda", generator=g) / math.sqrt(K)).bfloat16()
        Cs = torch.empty(M, N, device="cuda")
        ws = torch.empty(tg.gemm_splitk_workspace_size(M, N, K, 256) + 16, dtype=torch.uint8,
                         device="cuda")
        sh = torch.cuda.current_stream().cuda_stream
        emit("f4_plain", M, N, K, timeit(lambda: tg.matmul(A, B, out=Cs), 200))
        best = None
        for splits in (2, 4, 8, 16, 32, 64):
            ms = timeit(lambda: tg.gemm_splitk(A.data_ptr(), B.data_ptr(), Cs.data_ptr(), M, N, K,
                                               splits, tg.BF16, tg.F32, tg.F32, ws.data_ptr(),
                                               ws.numel(), sh), 200)
            if best is None or ms < best[1]:
                best = (splits, ms)
        emit("f4_splitk_best", M, N, K, best[1], splits=best[0])
    # whole waves vs the split last wave: interleaved rounds, so that heat and
    # power-cap drift over the run does not favour whichever variant runs first
    for m in (2560, 4096, 6144, 8192):
        A = (torch.randn(m, m, device="cuda", generator=g) / math.sqrt(m)).bfloat16()
        B = (torch.randn(m, m, device="cuda", generator=g) / math.sqrt(m)).bfloat16()
        Cb = torch.empty(m, m, device="cuda", dtype=torch.bfloat16)
        ws = torch.empty(tg.gemm_workspace_size(m, m, m), dtype=torch.uint8, device="cuda")
        steps = 100 if m <= 4096 else 30
        fns = {"f4_whole_waves": lambda: tg.matmul(A, B, out=Cb, out_dtype=torch.bfloat16),
               "f4_last_wave_split": lambda: tg.matmul_ws(A, B, out=Cb, workspace=ws)}
        rounds = {k: [] for k in fns}
        for _ in range(6):
            for k, f in fns.items():
                rounds[k].append(timeit(f, steps))
        for k in fns:
            emit(k, m, m, m, statistics.median(rounds[k]))


def main():
    args = parse_args()
    if args.sweep:
        run_sweep()
        return
    if args.rows:
        run_rows()
        return
    if args.simt:
        run_simt()
        return
    if args.small_sweep:
        run_small_sweep(args.sweep_shapes, args.sweep_calls)
        return
    world_env = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, rank, world_env)
        return
    rank, world, local = dist_setup(args.gpus)
    try:
        run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
