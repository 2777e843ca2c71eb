#!/usr/bin/env python3
"""Benchmark of the fused fp16 GEMM  C = GELU(A @ B + bias)  at M = N = K = 8192.

One step = one call of gemm_f16 (the whole path: TMA loads, tcgen05 MMA into
tensor memory, fused bias + erf-GELU epilogue, one fp16 write of C) on
seeded synthetic inputs already resident in HBM.  Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--layout nn|nt|tn|tt] [--no-cpu-baseline]

--layout stores A (first letter) and/or B (second) transposed in HBM, e.g.
"nt" = B held as N x K like a Linear layer's weight; the call is then
gemm_f16_ex with the matching flags.  The default "nn" is plain row-major.

--impl reference times the CPU oracle (fp64, all host cores) on bounded row
samples of the same workload: the comparison arm.  N > 1 runs independent
replicas, one per GPU (weak scaling; no collective on the data path).

The attention workloads (--workload attn_*) time attn_f16_fwd the same way:
one step = one attention forward over (B, H, S, D) inputs resident in HBM,
throughput by the FLOP model 4 B H S^2 D (halved when causal).
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "TFLOP/s and % of GB300 fp16 tensor peak for fused bias+GELU GEMM"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "fused8192"
L2_BYTES = 129 * 10 ** 6
FALLBACK_TENSOR_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
FP16_PER_BF16 = 1.0          # nominal dense fp16 rate / dense bf16 rate
KERNEL_SOURCES = ("dense_fp16_tensor_tma_gb300/csrc/gemm_kernels.cuh",
                  "dense_fp16_tensor_tma_gb300/csrc/gemm_kernels_pair.cuh",
                  "dense_fp16_tensor_tma_gb300/csrc/gemm_kernels_swap.cuh",
                  "dense_fp16_tensor_tma_gb300/csrc/ptx.cuh",
                  "dense_fp16_tensor_tma_gb300/csrc/gemm_f16.cu")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


ATTN_SOURCES = ("dense_fp16_tensor_tma_gb300/csrc/attn_kernels.cuh",
                "dense_fp16_tensor_tma_gb300/csrc/attn4_kernels.cuh",
                "dense_fp16_tensor_tma_gb300/csrc/attn2_kernels.cuh",
                "dense_fp16_tensor_tma_gb300/csrc/attn3_kernels.cuh",
                "dense_fp16_tensor_tma_gb300/csrc/attn_f16.cu",
                "dense_fp16_tensor_tma_gb300/csrc/ptx.cuh")


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


LAYOUT_TEXT = {"nn": "row-major A [M,K] and B [K,N]", "nt": "row-major A [M,K], B stored transposed [N,K]",
               "tn": "A stored transposed [K,M], row-major B [K,N]", "tt": "A stored [K,M] and B stored [N,K]"}


def workload_config(w, epi, layout="nn"):
    return {
        "workload": f"{w.name}: M={w.M} N={w.N} K={w.K} epilogue={epi}, fp16 {LAYOUT_TEXT[layout]} "
                    f"~{w.ab_dist}*{w.ab_scale}, bias ~{w.bias_dist}, seed {w.seed}",
        "M": w.M, "N": w.N, "K": w.K, "epilogue": epi, "seed": w.seed, "layout": layout,
        "accumulate": "f32", "flops_per_step": w.flops(), "alg_bytes_per_step": w.alg_bytes(),
        "l2": ("inputs larger than L2 (no flush)" if w.alg_bytes() > L2_BYTES
               else "L2 flushed between steps (256 MiB write)"),
    }


def attn_kernel_name(w, sms: int) -> str:
    """The attention kernel the library's plan picks for this workload (its
    host-only attn_f16_plan: the two-tile kernels for non-causal problems and
    for causal ones with a multiple of 4 tiles per head that split evenly, the
    one-tile kernel otherwise)."""
    import dense_fp16_tensor_tma_gb300 as g
    name = g.attn_f16_plan(w.B, w.H, w.S, w.D, w.causal, sms)["kernel_name"]
    return f"{name}<{w.D}>"


def kernel_name(plan):
    """Name of the tensor-core kernel a plan launches."""
    if plan.get("path") == 3:
        return f"gemm_f16_swap_kernel<{plan['tile_m']}, {plan['stages']}> (swap-AB)"
    if plan.get("path") != 2:
        return "gemm_f16_bias_only_kernel"
    if plan.get("tile_m") == 256:
        return f"gemm_f16_tc2_kernel (CTA pair, 256x256, {plan['stages']} stages)"
    return f"gemm_f16_tc_kernel<{plan['tile_n']}, {plan['stages']}>"


# A timed window at least this long runs under the board's power cap (the
# clock record of a 1000-step 8192^3 run shows sw_power_cap within it), so its
# kernels are measured against the sustained tensor peak; shorter windows
# against the burst peak.
SUSTAINED_WINDOW_S = 0.25
FALLBACK_TENSOR_SUSTAINED_TFLOPS = 1700.0


def read_peaks(window_s=0.0):
    """(fp16 tensor TFLOP/s, HBM GB/s, source): the measured figures (the
    sustained tensor peak for a timed window of SUSTAINED_WINDOW_S or more,
    else the burst one), else the fallbacks."""
    sustained = window_s >= SUSTAINED_WINDOW_S
    kind = "sustained" if sustained else "burst"
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        tflops = float(pk["bf16_tflops_sustained" if sustained else "bf16_tflops"])
        return tflops * FP16_PER_BF16, float(pk["hbm_gbs"]), f"measured bf16 {kind}"
    except (OSError, KeyError, ValueError):
        tflops = FALLBACK_TENSOR_SUSTAINED_TFLOPS if sustained else FALLBACK_TENSOR_TFLOPS
        return tflops, FALLBACK_HBM_GBS, f"fallback {kind}"


def roofline(w, avg_launch_ms, traffic, plan, window_s):
    """Roofline of the dominant kernel: tensor-bound when the workload's
    arithmetic intensity (algorithmic FLOPs per algorithmic byte) is above the
    ridge point of the two peaks, else HBM-bound.  window_s: the timed
    window's length (selects the burst or sustained tensor peak)."""
    tensor_peak, hbm_peak, src = read_peaks(window_s)
    intensity = w.flops() / w.alg_bytes()
    ridge = tensor_peak * 1e12 / (hbm_peak * 1e9)
    if intensity >= ridge:
        achieved, peak, unit, bound = w.flops() / (avg_launch_ms * 1e-3) / 1e12, tensor_peak, "TFLOP/s", "tensor"
        peak_src = f"{src} (x fp16/bf16 ratio {FP16_PER_BF16})"
    else:
        achieved, peak, unit, bound = w.alg_bytes() / (avg_launch_ms * 1e-3) / 1e9, hbm_peak, "GB/s", "hbm"
        peak_src = f"{src} (copy bandwidth)"
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "traffic": traffic, "peak_source": peak_src, "intensity_flop_per_byte": intensity,
            "ridge_flop_per_byte": ridge, "kernel": kernel_name(plan), "avg_launch_ms": avg_launch_ms}


def committed_traffic(workload_name, sources=KERNEL_SOURCES):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload_name)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("kernel_source_hash") != kernel_source_hash(sources):
        return None
    return rec.get("dram_bytes_per_launch")


def launch_stats(per_launch_ms):
    """Median, min, p90 and mean of the per-launch CUDA-event times (ms): the
    median-of-reps timing of "TileLang: Write, Autotune, and Ship Fused
    Tensor-Core Kernels from Python", Practical defaults, with its spread."""
    xs = sorted(per_launch_ms)
    p90 = xs[min(len(xs) - 1, int(math.ceil(0.9 * len(xs))) - 1)]
    return {"median": statistics.median(xs), "min": xs[0], "p90": p90, "mean": statistics.mean(xs),
            "n": len(xs)}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid=None, interval_ms=20):
        self.proc = None
        self.lines = []
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", str(interval_ms)]
        if gpu_uuid:
            cmd += ["-i", gpu_uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        self.t_start = time.time()

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return [l for l in out.splitlines() if l.strip()]

    @staticmethod
    def parse(lines):
        """[(unix_time, sm_mhz, sm_max_mhz, set(active reasons))]"""
        out = []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                sm, smax = float(parts[2]), float(parts[3])
            except (ValueError, IndexError):
                continue
            out.append((ts, sm, smax, {n for n, v in zip(names, parts[6:10]) if v.lower() == "active"}))
        return out

    @staticmethod
    def summarize(samples, t0=None, t1=None, pad_s=0.03):
        """Median SM clock and throttle reasons of the samples inside [t0-pad, t1+pad];
        when the window holds none (a short run), the samples of the whole run."""
        window = "timed"
        sel = samples
        if t0 is not None and t1 is not None:
            sel = [s for s in samples if t0 - pad_s <= s[0] <= t1 + pad_s]
            if not sel:
                sel, window = samples, "whole run (timed window shorter than the sampling interval)"
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": window}
        reasons = set().union(*[s[3] for s in sel])
        return {"sm_mhz": statistics.median(s[1] for s in sel), "sm_max_mhz": sel[-1][2],
                "reasons": sorted(reasons), "samples": len(sel), "window": window}


# ------------------------------------------------------------------ distributed (replicas)

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    return world, rank, local


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(world, x: float) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ end-to-end steps

E2E_MODE = ("pipelined: step i's host-to-device copies overlap step i-1's computation and step i-2's "
            "device-to-host copy (two device buffer sets, three streams); serial_*: copy in, compute, copy out "
            "one after another on one stream")


def pipelined_e2e(torch, dev, world, nsteps, comp_stream, copy_in, compute, copy_out):
    """End-to-end steps the way a serving loop runs them: step i's inputs are
    copied from pinned host memory into one of two device buffer sets on a
    copy-in stream while step i - 1 computes on `comp_stream` and step i - 2's
    result is copied out on a copy-out stream.  A set's inputs are overwritten
    only after the step that read them has computed, and its result only after
    it has been copied out.  Every step's copies lie inside the timed region
    (first copy-in to last copy-out).  copy_in(b), compute(b), copy_out(b) enqueue
    on the current stream for buffer set b.  Returns milliseconds (max over ranks)."""
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)

    def run(n):
        ev_in, ev_comp, ev_out = [], [], []
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[i - 2])
                copy_in(b)
                ev_in.append(torch.cuda.Event())
                ev_in[-1].record(s_in)
            with torch.cuda.stream(comp_stream):
                comp_stream.wait_event(ev_in[i])
                if i >= 2:
                    comp_stream.wait_event(ev_out[i - 2])
                compute(b)
                ev_comp.append(torch.cuda.Event())
                ev_comp[-1].record(comp_stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[i])
                copy_out(b)
                ev_out.append(torch.cuda.Event())
                ev_out[-1].record(s_out)

    run(3)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist_barrier(world)
    torch.cuda.synchronize(dev)
    ev0.record(s_in)
    run(nsteps)
    ev1.record(s_out)                  # the last copy-out depends on every earlier operation
    torch.cuda.synchronize(dev)
    ms = dist_max(world, ev0.elapsed_time(ev1))
    dist_barrier(world)
    return ms


# ------------------------------------------------------------------ CPU oracle timing

def oracle_rows_timing(w, epi, A, B, bias, target_s):
    """Time the oracle on a bounded sample of full rows; returns (tflops, seconds, rows, threads)."""
    import oracle
    b = bias if epi != "none" else None
    threads = oracle.default_threads()
    # two probes separate the per-call operand conversion from the per-row cost
    p1 = max(1, min(w.M, threads))
    p2 = max(p1, min(w.M, 4 * threads))
    t0 = time.perf_counter()
    oracle.gemm_rows(A, B, b, epi, np.arange(p1))
    t1 = time.perf_counter()
    oracle.gemm_rows(A, B, b, epi, np.arange(p2))
    t2 = time.perf_counter()
    per_row = max((t2 - t1) - (t1 - t0), 1e-6) / max(1, p2 - p1)
    rows = int(min(w.M, max(p2, target_s / per_row)))
    rows = min(w.M, max(threads, rows // threads * threads))
    t0 = time.perf_counter()
    oracle.gemm_rows(A, B, b, epi, np.arange(rows))
    dt = time.perf_counter() - t0
    return 2.0 * rows * w.N * w.K / dt / 1e12, dt, rows, threads


def run_reference(args, w, epi):
    world, rank, _ = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    A, B, bias = w.make()
    b = bias if epi != "none" else None
    threads = oracle.default_threads()
    # calibrate rows per step so the whole run stays within a few minutes
    t0 = time.perf_counter()
    oracle.gemm_rows(A, B, b, epi, np.arange(min(w.M, threads)))
    per_row = (time.perf_counter() - t0) / min(w.M, threads)
    budget_s = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    rows_per_step = int(min(w.M, max(1, budget_s / max(per_row, 1e-9))))
    rows_per_step = max(1, min(w.M, rows_per_step // threads * threads or rows_per_step))
    for i in range(args.warmup):
        oracle.gemm_rows(A, B, b, epi, (np.arange(rows_per_step) + i * rows_per_step) % w.M)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.gemm_rows(A, B, b, epi, (np.arange(rows_per_step) + i * rows_per_step) % w.M)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows_per_step * w.N * w.K * args.steps
    value = flops / dt / 1e12
    sample = (f"{rows_per_step} of {w.M} output rows per step (full K={w.K} dot products, all N={w.N} "
              f"columns, epilogue {epi}), fp64 C++ oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, epi, args.layout),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm

def run_ours(args, w, epi):
    import torch
    world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import dense_fp16_tensor_tma_gb300 as g

    props = torch.cuda.get_device_properties(dev)
    # replicas: each rank owns an independent problem of the same shape
    wr = w if world == 1 else workloads.Workload(**{**w.__dict__, "seed": w.seed + 1000 * rank})
    t_gen = time.perf_counter()
    A, B, bias = wr.make()
    log(f"[rank {rank}] inputs generated in {time.perf_counter() - t_gen:.1f}s")
    b_np = bias if epi != "none" else None
    ta, tbt = args.layout[0] == "t", args.layout[1] == "t"
    # the operands as stored in HBM (the same logical matrices)
    A_st = np.ascontiguousarray(A.T) if ta else A
    B_st = np.ascontiguousarray(B.T) if tbt else B
    lda, ldb, flags = A_st.shape[1], B_st.shape[1], (1 if ta else 0) | (2 if tbt else 0)
    tA = torch.from_numpy(A_st).to(dev)
    tB = torch.from_numpy(B_st).to(dev)
    tb = torch.from_numpy(b_np).to(dev) if b_np is not None else None
    C = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    flush = None
    if w.alg_bytes() <= L2_BYTES:
        flush = torch.empty(256 * 2 ** 20 // 4, dtype=torch.float32, device=dev)
    plan = g.gemm_f16_plan(w.M, w.N, w.K, epi, num_sms=props.multi_processor_count,
                           a_addr=tA.data_ptr(), b_addr=tB.data_ptr(), c_addr=C.data_ptr(),
                           bias_addr=tb.data_ptr() if tb is not None else 0, lda=lda, ldb=ldb,
                           trans_a=ta, trans_b=tbt)
    launches_per_step = 1 + plan["pack_a"] + plan["pack_b"]

    def flush_l2():
        if flush is not None:
            flush.fill_(1.0)

    def step():
        st = g.gemm_f16_ex_ptr(tA.data_ptr(), lda, tB.data_ptr(), ldb, tb.data_ptr() if tb is not None else 0,
                               C.data_ptr(), w.N, w.M, w.N, w.K, epi, flags, sh)
        if st != 0:
            raise g.GemmError(st)

    uuid = None
    try:
        uuid = "GPU-" + str(props.uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            flush_l2()
            step()
    stream.synchronize()
    st, word = g.gemm_f16_debug_status(stream)
    if st != 0:
        raise SystemExit(f"device status {st} ({word:#x}) after warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    dist_barrier(world)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush_l2()                 # outside the events: only the GEMM is timed
            starts[i].record(stream)
            step()
            ends[i].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    dist_barrier(world)
    clock_lines = sampler.stop()
    per_launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    # back to back (inputs larger than L2): the whole window; with an L2 flush
    # between steps: the sum of the per-step windows, which exclude the flush
    elapsed_ms = starts[0].elapsed_time(ends[-1]) if flush is None else sum(per_launch_ms)
    elapsed_ms = dist_max(world, elapsed_ms)
    st, word = g.gemm_f16_debug_status(stream)
    if st != 0:
        raise SystemExit(f"device status {st} ({word:#x}) after timed steps")

    flops = w.flops()
    value = world * flops * args.steps / (elapsed_ms * 1e-3) / 1e12
    avg_launch_ms = statistics.mean(per_launch_ms)
    traffic = committed_traffic(w.name if args.layout == "nn" else f"{w.name}:{args.layout}")
    roof = roofline(w, avg_launch_ms, traffic, plan, elapsed_ms * 1e-3)
    tensor_peak = read_peaks(elapsed_ms * 1e-3)[0]

    # ---- end to end: pinned host buffers through the C ABI, copies inside the timed region
    hA = torch.from_numpy(A_st).pin_memory()
    hB = torch.from_numpy(B_st).pin_memory()
    hb = torch.from_numpy(b_np).pin_memory() if b_np is not None else None
    hC = torch.empty((w.M, w.N), dtype=torch.float16).pin_memory()
    h2d = hA.numel() * 2 + hB.numel() * 2 + (hb.numel() * 2 if hb is not None else 0)
    d2h = hC.numel() * 2

    def e2e_step():
        tA.copy_(hA, non_blocking=True)
        tB.copy_(hB, non_blocking=True)
        if hb is not None:
            tb.copy_(hb, non_blocking=True)
        step()
        hC.copy_(C, non_blocking=True)

    e2e_steps = args.steps
    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
    stream.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist_barrier(world)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    serial_ms = dist_max(world, ev0.elapsed_time(ev1))
    dist_barrier(world)
    serial_value = world * flops * e2e_steps / (serial_ms * 1e-3) / 1e12
    # the same steps pipelined over two device buffer sets (copies overlap computation)
    sets_A, sets_B = [tA, torch.empty_like(tA)], [tB, torch.empty_like(tB)]
    sets_b = [tb, torch.empty_like(tb)] if tb is not None else [None, None]
    sets_C, host_C = [C, torch.empty_like(C)], [hC, torch.empty_like(hC).pin_memory()]

    def copy_in(b):
        sets_A[b].copy_(hA, non_blocking=True)
        sets_B[b].copy_(hB, non_blocking=True)
        if hb is not None:
            sets_b[b].copy_(hb, non_blocking=True)

    def compute(b):
        st = g.gemm_f16_ex_ptr(sets_A[b].data_ptr(), lda, sets_B[b].data_ptr(), ldb,
                               sets_b[b].data_ptr() if sets_b[b] is not None else 0, sets_C[b].data_ptr(), w.N,
                               w.M, w.N, w.K, epi, flags, torch.cuda.current_stream().cuda_stream)
        if st != 0:
            raise g.GemmError(st)

    def copy_out(b):
        host_C[b].copy_(sets_C[b], non_blocking=True)

    e2e_ms = pipelined_e2e(torch, dev, world, e2e_steps, stream, copy_in, compute, copy_out)
    e2e_value = world * flops * e2e_steps / (e2e_ms * 1e-3) / 1e12
    st, word = g.gemm_f16_debug_status(stream)
    if st != 0:
        raise SystemExit(f"device status {st} ({word:#x}) after the end-to-end steps")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tfl, secs, rows, threads = oracle_rows_timing(w, epi, A, B, bias, target_s=args.cpu_seconds)
        cpu = {"value": tfl, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{rows} of {w.M} output rows (full N, full K), fp64 C++ oracle, {secs:.1f}s"}

    if rank == 0:
        clocks = ClockSampler.summarize(ClockSampler.parse(clock_lines), t_wall0, t_wall1)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": elapsed_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic",
            "config": {**workload_config(w, epi, args.layout),
                       "parallelism": f"replicas{world}" if world > 1 else "single"},
            "pct_of_peak": 100.0 * (flops / (avg_launch_ms * 1e-3) / 1e12) / tensor_peak,
            "launch_ms": launch_stats(per_launch_ms),
            "roofline": roof,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms / e2e_steps, "steps": e2e_steps,
                    "mode": E2E_MODE, "serial_value": serial_value, "serial_ms_per_step": serial_ms / e2e_steps},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                       "reasons": clocks["reasons"], "samples": clocks["samples"],
                       "window": clocks["window"], "window_s": round(t_wall1 - t_wall0, 3)},
            "cpu_baseline": cpu,
            "plan": plan,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ attention forward

ATTN_METRIC = "TFLOP/s of fused fp16 attention forward (FLOP model 4 B H S^2 D, halved when causal)"


def attn_config(w):
    return {
        "workload": f"{w.name}: B={w.B} H={w.H} S={w.S} D={w.D} causal={int(w.causal)}, fp16 Q,K,V ~normal, "
                    f"scale 1/sqrt(D), seed {w.seed}",
        "B": w.B, "H": w.H, "S": w.S, "D": w.D, "causal": w.causal, "seed": w.seed,
        "flops_per_step": w.flops(), "alg_bytes_per_step": w.alg_bytes(),
        "flop_model": "4 B H S^2 D, x0.5 causal",
        "l2": ("inputs larger than L2 (no flush)" if w.alg_bytes() > L2_BYTES
               else "L2 flushed between steps (256 MiB write)"),
    }


def attn_oracle_timing(w, Q, K, V, target_s):
    """Time the oracle on a bounded sample of query rows; (TFLOP/s by the FLOP model, s, rows, threads)."""
    import oracle
    threads = oracle.default_threads()
    scale = 1.0 / math.sqrt(w.D)
    probe = w.sample_rows(max(threads, 16))
    t0 = time.perf_counter()
    oracle.attention_rows(Q, K, V, w.causal, scale, probe)
    per_row = max(time.perf_counter() - t0, 1e-6) / probe.size
    total = w.B * w.H * w.S
    n = int(min(total, max(threads, target_s / per_row)))
    rows = w.sample_rows(n)
    t0 = time.perf_counter()
    oracle.attention_rows(Q, K, V, w.causal, scale, rows)
    dt = time.perf_counter() - t0
    # model FLOPs of the sampled rows: the workload's FLOPs x the share of rows
    return w.flops() * rows.size / total / dt / 1e12, dt, rows.size, threads


def run_attention_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    Q, K, V = w.make()
    budget_s = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    tfl, _, rows, threads = attn_oracle_timing(w, Q, K, V, budget_s)
    total = w.B * w.H * w.S
    sample_rows = w.sample_rows(rows)
    scale = 1.0 / math.sqrt(w.D)
    for _ in range(args.warmup):
        oracle.attention_rows(Q, K, V, w.causal, scale, sample_rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention_rows(Q, K, V, w.causal, scale, sample_rows)
    dt = time.perf_counter() - t0
    value = w.flops() * sample_rows.size / total * args.steps / dt / 1e12
    sample = (f"{sample_rows.size} of {total} query rows per step (every admissible key, full D), "
              f"fp64 C++ oracle")
    line = {
        "impl": "reference", "metric": ATTN_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": attn_config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_attention(args, w):
    import torch
    world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import dense_fp16_tensor_tma_gb300 as g

    wr = w if world == 1 else workloads.AttnWorkload(**{**w.__dict__, "seed": w.seed + 1000 * rank})
    t_gen = time.perf_counter()
    Q, K, V = wr.make()
    log(f"[rank {rank}] inputs generated in {time.perf_counter() - t_gen:.1f}s")
    tq, tk, tv = (torch.from_numpy(x).to(dev) for x in (Q, K, V))
    O = torch.empty_like(tq)
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    flush = torch.empty(256 * 2 ** 20 // 4, dtype=torch.float32, device=dev) if w.alg_bytes() <= L2_BYTES else None

    def step():
        st = g.attn_f16_fwd_ptr(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), O.data_ptr(), w.B, w.H, w.S, w.D,
                                w.causal, 0.0, sh)
        if st != 0:
            raise g.GemmError(st, "attn_f16_fwd")

    props = torch.cuda.get_device_properties(dev)
    uuid = None
    try:
        uuid = "GPU-" + str(props.uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            if flush is not None:
                flush.fill_(1.0)
            step()
    stream.synchronize()
    st, word = g.attn_f16_debug_status(stream)
    if st != 0:
        raise SystemExit(f"device status {st} ({word:#x}) after warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    dist_barrier(world)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            if flush is not None:
                flush.fill_(1.0)       # outside the events
            starts[i].record(stream)
            step()
            ends[i].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    dist_barrier(world)
    clock_lines = sampler.stop()
    per_launch_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    elapsed_ms = starts[0].elapsed_time(ends[-1]) if flush is None else sum(per_launch_ms)
    elapsed_ms = dist_max(world, elapsed_ms)
    st, word = g.attn_f16_debug_status(stream)
    if st != 0:
        raise SystemExit(f"device status {st} ({word:#x}) after timed steps")
    flops = w.flops()
    value = world * flops * args.steps / (elapsed_ms * 1e-3) / 1e12
    avg_launch_ms = statistics.mean(per_launch_ms)
    tensor_peak, _, src = read_peaks(elapsed_ms * 1e-3)
    achieved = flops / (avg_launch_ms * 1e-3) / 1e12
    traffic = committed_traffic(w.name, ATTN_SOURCES)
    roof = {"bound": "tensor", "achieved": achieved, "peak": tensor_peak, "unit": "TFLOP/s",
            "frac": achieved / tensor_peak, "traffic": traffic,
            "peak_source": f"{src} (x fp16/bf16 ratio {FP16_PER_BF16})",
            "kernel": attn_kernel_name(w, props.multi_processor_count), "avg_launch_ms": avg_launch_ms}

    # ---- end to end: pinned host Q, K, V in and O out through the C ABI every step
    hq, hk, hv = (torch.from_numpy(x).pin_memory() for x in (Q, K, V))
    ho = torch.empty(tuple(O.shape), dtype=torch.float16).pin_memory()
    h2d = 3 * hq.numel() * 2
    d2h = ho.numel() * 2

    def e2e_step():
        tq.copy_(hq, non_blocking=True)
        tk.copy_(hk, non_blocking=True)
        tv.copy_(hv, non_blocking=True)
        step()
        ho.copy_(O, non_blocking=True)

    e2e_steps = max(1, min(args.steps, 50))
    with torch.cuda.stream(stream):
        for _ in range(2):
            e2e_step()
    stream.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist_barrier(world)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    serial_ms = dist_max(world, ev0.elapsed_time(ev1))
    dist_barrier(world)
    serial_value = world * flops * e2e_steps / (serial_ms * 1e-3) / 1e12
    # the same steps pipelined over two device buffer sets (copies overlap computation)
    sets = [(tq, tk, tv, O), tuple(torch.empty_like(x) for x in (tq, tk, tv, O))]
    host_O = [ho, torch.empty_like(ho).pin_memory()]

    def copy_in(b):
        for d, h in zip(sets[b][:3], (hq, hk, hv)):
            d.copy_(h, non_blocking=True)

    def compute(b):
        q_, k_, v_, o_ = sets[b]
        st = g.attn_f16_fwd_ptr(q_.data_ptr(), k_.data_ptr(), v_.data_ptr(), o_.data_ptr(), w.B, w.H, w.S, w.D,
                                w.causal, 0.0, torch.cuda.current_stream().cuda_stream)
        if st != 0:
            raise g.GemmError(st, "attn_f16_fwd")

    def copy_out(b):
        host_O[b].copy_(sets[b][3], non_blocking=True)

    e2e_ms = pipelined_e2e(torch, dev, world, e2e_steps, stream, copy_in, compute, copy_out)
    e2e_value = world * flops * e2e_steps / (e2e_ms * 1e-3) / 1e12
    st, word = g.attn_f16_debug_status(stream)
    if st != 0:
        raise SystemExit(f"device status {st} ({word:#x}) after the end-to-end steps")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tfl, secs, rows, threads = attn_oracle_timing(w, Q, K, V, args.cpu_seconds)
        cpu = {"value": tfl, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{rows} of {w.B * w.H * w.S} query rows (every admissible key, full D), fp64 C++ oracle, "
                         f"{secs:.1f}s"}
    if rank == 0:
        clocks = ClockSampler.summarize(ClockSampler.parse(clock_lines), t_wall0, t_wall1)
        line = {
            "metric": ATTN_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": elapsed_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic",
            "config": {**attn_config(w), "parallelism": f"replicas{world}" if world > 1 else "single"},
            "launch_ms": launch_stats(per_launch_ms),
            "roofline": roof,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms / e2e_steps, "steps": e2e_steps,
                    "mode": E2E_MODE, "serial_value": serial_value, "serial_ms_per_step": serial_ms / e2e_steps},
            "gpu_launches": args.steps,
            "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                       "reasons": clocks["reasons"], "samples": clocks["samples"],
                       "window": clocks["window"], "window_s": round(t_wall1 - t_wall0, 3)},
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(workloads.WORKLOADS) + sorted(workloads.ATTN_WORKLOADS))
    ap.add_argument("--epilogue", default=None)
    ap.add_argument("--layout", default="nn", choices=sorted(LAYOUT_TEXT))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.steps < 1:
        raise SystemExit("--steps must be >= 1")
    if args.workload in workloads.ATTN_WORKLOADS:
        w = workloads.ATTN_WORKLOADS[args.workload]
        return run_attention_reference(args, w) if args.impl == "reference" else run_attention(args, w)
    w = workloads.WORKLOADS[args.workload]
    epi = args.epilogue or w.epilogues[-1]
    if args.impl == "reference":
        return run_reference(args, w, epi)
    return run_ours(args, w, epi)


if __name__ == "__main__":
    sys.exit(main())
