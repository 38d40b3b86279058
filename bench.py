#!/usr/bin/env python3
"""Benchmark of the exact-sum GEMM on GB300.

Workload (one "step"): the exact GEMM C = RNE_f32(A B^T) at M = N = K = 4096,
f32, A and B iid N(0,1) from seed 0 (rank r uses seed r), with inputs resident
in HBM; between steps a 256 MiB buffer is written to flush the 129 MB L2.
Metric: exact-GEMM GFLOP/s = 2 M N K / t (whole job, summed over ranks).

Printed as one JSON line on rank 0, with:
  roofline      dominant kernel vs the integer-ALU issue peak
  cpu_baseline  the CPU oracle on a bounded row sample of the same workload
  e2e           the same metric through the public API from pinned host
                buffers, copies included
  clocks        nvidia-smi SM clocks and throttle reasons during the timed region
  sharded       2-way K-sharded partial/combine/finalize of the same GEMM, with
                the combine and finalize kernels' HBM rooflines

``--impl reference`` times the CPU oracle instead (the reference arm).
Multi-GPU: launched with torchrun, every rank runs its own independent
problem (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "exact-GEMM GFLOP/s (2MNK/s) at 4096^3 f32"
UNIT = "GFLOP/s"
M = N = K = 4096
FLUSH_BYTES = 256 << 20
SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASON_NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
DTYPE_DETAIL = ("inputs and output f32; products of bf16 residues (|r| <= 138) on the tensor "
                "cores with exact fp32 accumulation, reduced modulo p; int64 CRT rebuild and "
                "one rounding (the digits are exact integers throughout)")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=["normal", "wide", "loguniform100"], default="normal",
                   help="normal: N(0,1) (the headline); wide: |x| = 2^U[-40,40]; "
                        "loguniform100: |x| = 2^U[-100,100] (beyond the wide path's window: "
                        "the general kernel; with --mnk, for profiling)")
    p.add_argument("--cpu-rows", type=int, default=512,
                   help="rows of the 4096^3 problem the CPU baseline samples")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the e2e, sharded and CPU-baseline measurements")
    p.add_argument("--configs", action="store_true",
                   help="time each workload configuration (one JSON line each) instead of "
                        "the headline run")
    p.add_argument("--op", choices=["gemm", "partial", "batched"], default="gemm",
                   help="the timed call: det_gemm (the headline), det_gemm_partial into a "
                        "preallocated digit array (for profiling the digit write-out), or "
                        "det_gemm_strided_batched over --batch entries of M x N x K (default "
                        "128 x 128 x 4096; for profiling the batched pipeline)")
    p.add_argument("--batch", type=int, default=64, help="entries of --op batched")
    p.add_argument("--mnk", type=int, nargs=3, default=None, metavar=("M", "N", "K"),
                   help="override the problem size (profiling of small cases only)")
    args = p.parse_args()
    global M, N, K
    if args.mnk:
        M, N, K = args.mnk
    elif args.op == "batched":
        M, N, K = 128, 128, 4096
    return args


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value, dist, device):
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(rank):
    """Each rank runs its own independent problem: seed = rank."""
    return int(rank)


def make_inputs(seed, workload):
    from exact_sum_gemm_gb300 import workloads as wl
    if workload == "normal":
        return wl.normal_f32((M, K), seed, 0), wl.normal_f32((N, K), seed, 1)
    span = 40 if workload == "wide" else 100
    return (wl.loguniform_f32((M, K), seed, 0, lo=-span, hi=span),
            wl.loguniform_f32((N, K), seed, 1, lo=-span, hi=span))


def workload_config(workload, extra=None):
    dist = {"normal": "iid N(0,1)", "wide": "|x|=2^U[-40,40]",
            "loguniform100": "|x|=2^U[-100,100]"}[workload]
    cfg = {"workload": f"det_gemm f32 M={M} N={N} K={K}, A,B {dist}, seed 0",
           "M": M, "N": N, "K": K, "dtype_in": "f32", "dtype_out": "f32",
           "l2": "flushed: 256 MiB write between steps (outside the per-step events)",
           "inputs": "resident in HBM (e2e: copied from pinned host memory every step)"}
    if extra:
        cfg.update(extra)
    return cfg


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    def __init__(self, uuid=None):
        self.proc = None
        self.uuid = uuid

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={SMI_FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(REASON_NAMES, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- helpers

def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def cpu_baseline(workload, rows, seed=0):
    """The oracle, as it stands, on `rows` rows of the same problem (all host cores)."""
    import oracle
    oracle.build()
    A, B = make_inputs(seed, workload)
    sel = np.linspace(0, M - 1, rows).astype(np.int64)
    A_s = np.ascontiguousarray(A[sel])
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle.gemm(A_s, B, nthreads=cores)
    dt = time.perf_counter() - t0
    return {"value": round(2.0 * rows * N * K / dt / 1e9, 4), "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"{rows} evenly spaced rows of the 4096^3 problem ({rows}x4096x4096 "
                      f"exact MACs), {dt:.2f} s wall on {cores} threads"}


# Per-launch DRAM traffic of the dominant kernel, from one ncu capture of this
# benchmark's full-size workload (profiles/residue_gemm_kernel_f32_4096.md).
# Reported only while the kernel's sources still hash to the captured
# fingerprint; otherwise "traffic" is null.
CAPTURED_TRAFFIC = {
    # det_gemm at 4096^3 runs the tensor-core kernel once per row band (two
    # bands of 2816 and 1280 rows); bytes are per launch, the mean of the
    # call's two launches
    "residue_gemm": {"fingerprint": "93aec01f9a9bf60e", "mnk": (4096, 4096, 4096),
                     "workload": "normal", "launches_per_call": 2,
                     "bytes": (982269696 + 130824704 + 697994752 + 52084992) // 2},
}
KERNEL_SOURCES = {
    "residue_gemm": ["gemm_tc2.cu", "gemm_tc.cu", "tc_ptx.cuh", "det_residue.cuh"],
}


def kernel_fingerprint(stage):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(stage, []):
        with open(os.path.join(ROOT, "exact_sum_gemm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def captured_traffic(stage, workload):
    """(bytes per launch, launches per call) of the capture, or (None, None)."""
    rec = CAPTURED_TRAFFIC.get(stage)
    if not rec or rec["mnk"] != (M, N, K) or rec["workload"] != workload:
        return None, None
    if kernel_fingerprint(stage) != rec["fingerprint"]:
        return None, rec.get("launches_per_call")
    return rec["bytes"], rec.get("launches_per_call")


def stage_spans(timeline, calls):
    """{stage: (ms per call covered by its records, records per call)}.

    A record runs from when its stream reaches it to when its last kernel
    ends.  Records of one stage overlap where row bands run on two streams
    (the second band's tensor-core launch is enqueued while the first still
    runs and starts on the SMs the first one frees), so the covered time, the
    union of the intervals, is the stage's busy time; calls do not overlap."""
    by = {}
    for name, t0, t1 in timeline:
        by.setdefault(name, []).append((t0, t1))
    out = {}
    for name, iv in by.items():
        iv.sort()
        total, (cs, ce) = 0.0, iv[0]
        for t0, t1 in iv[1:]:
            if t0 > ce:
                total += ce - cs
                cs, ce = t0, t1
            else:
                ce = max(ce, t1)
        total += ce - cs
        out[name] = (total / calls, len(iv) / calls)
    return out


def roofline_for(stage_ms, stages, props, peaks, lib, workload="normal", pipes=None):
    """Roofline of the dominant stage (by device time per step)."""
    if not stage_ms:
        return None
    dom = max(stage_ms, key=stage_ms.get)
    t = stage_ms[dom] * 1e-3
    exact_flops = 2.0 * M * N * K
    if dom == "residue_gemm":
        # moduli per row band as the last call chose them (the two bands of a
        # 4096-row C hold 2048 rows each); the planes are written for the
        # worst-case count
        used = (ctypes.c_int * 8)()
        nb = lib.det_moduli_used(used, 8)
        worst = lib.det_residue_moduli(0, K)
        counts = list(used[:nb]) if nb > 0 else [worst]
        nmod = sum(counts) / len(counts)
        kp = (K + 63) // 64 * 64
        executed = 2.0 * M * N * kp * nmod
        peak = float(peaks.get("bf16_tflops", 1900.0))
        achieved = exact_flops / t / 1e12
        traffic, launches = captured_traffic(dom, workload)
        launches = launches or 1
        return {"kernel": "residue_gemm_pair_kernel (tcgen05 cta_group::2 bf16, 256x256 tiles)", "bound": "tensor",
                "achieved": round(achieved, 3), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 5), "traffic": traffic,
                "launches_per_call": launches,
                "traffic_algorithmic": int((nmod * (M + N * launches) * kp * 2 + nmod * M * N)
                                           // launches),
                "moduli_planes_written": worst,
                "peak_source": "MEASURED_PEAKS.json bf16_tflops (burst, measured)",
                "achieved_basis": "algorithmic exact flops 2MNK per call / the time the "
                                  "call's tensor-core launches cover (first start to last "
                                  "end; the two band launches overlap where the second "
                                  "takes the SMs the first frees)",
                "moduli": counts,
                "executed_tensor_tflops": round(executed / t / 1e12, 2),
                "executed_frac": round(executed / t / 1e12 / peak, 4),
                "kernel_ms": round(stage_ms[dom], 4)}
    return alu_roofline(dom, exact_flops / 2.0, stage_ms[dom], pipes)


def alu_roofline(kernel, macs, ms, pipes):
    """A CUDA-core exact kernel against the measured INT32 issue peak: exact
    MACs per second over instructions per second (one per MAC is the bound)."""
    achieved = macs / (ms * 1e-3) / 1e9
    if pipes:
        peak = max(pipes["kinds"]["iadd"]["gops"], pipes["kinds"]["lop3"]["gops"])
        src = "measured in this run: max(iadd, lop3) instructions/s (pipe_peaks)"
    else:
        peak = alu_peak_gops(152, 2070.0) / 2.0
        src = "fallback: 152 SMs x 128 lanes x 2070 MHz (no measurement in this run)"
    return {"kernel": kernel, "bound": "alu", "achieved": round(achieved, 3), "peak": peak,
            "unit": "G exact MAC/s vs G instr/s", "frac": round(achieved / peak, 5),
            "traffic": None, "peak_source": src, "kernel_ms": round(ms, 4)}


PIPE_KINDS = {"iadd": 0, "lop3": 1, "imad": 2, "imad_wide": 3, "ffma": 4, "dfma": 5}


def measure_pipe_peaks(lib, dev, uuid=None, target_s=0.6):
    """Measured throughput of the CUDA-core pipes an exact accumulation could
    run on: one launch per instruction kind (det_pipe_benchmark: 8 blocks of
    256 threads per SM, dependency rings of 8 accumulators per thread), timed
    with CUDA events over a launch of about `target_s` seconds after a short
    calibration launch; nvidia-smi samples the SM clock meanwhile."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    threads = lib.det_pipe_benchmark_threads_per_block()
    per_iter = lib.det_pipe_benchmark_ops_per_thread_iter()
    blocks = sms * 8
    out = torch.empty(blocks * threads, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    res = {}

    def timed(kind, iters):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        st = lib.det_pipe_benchmark(kind, iters, blocks, out.data_ptr(), stream.cuda_stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if st != 0:
            raise RuntimeError(f"det_pipe_benchmark({kind}) returned {st}")
        return e0.elapsed_time(e1) * 1e-3

    for name, kind in PIPE_KINDS.items():
        iters = 256
        t = timed(kind, iters)
        while t < 0.05:                      # calibrate on a launch long enough to time
            iters *= 4
            t = timed(kind, iters)
        iters = max(iters, int(iters * target_s / t))
        t = timed(kind, iters)
        ops = float(iters) * per_iter * threads * blocks
        res[name] = {"gops": round(ops / t / 1e9, 1), "seconds": round(t, 3),
                     "per_sm_per_clk": None}
    clocks = sampler.stop()
    mhz = clocks["sm_mhz"] if clocks else None
    for r in res.values():
        if mhz:
            r["per_sm_per_clk"] = round(r["gops"] * 1e9 / (sms * mhz * 1e6), 2)
    return {"kinds": res, "sms": sms, "clocks": clocks,
            "how": "det_pipe_benchmark: one launch per kind, 8 x 256 threads per SM, rings of 8 "
                   "independent accumulators, one PTX instruction per operation; ops / CUDA-event "
                   "time of a launch of about 0.6 s"}


def pipe_fractions(gflops, pipes):
    """The metric's reference pipes, from the measured peaks: exact MACs per
    second (GFLOP/s / 2) against the INT32 issue peak (the faster of the
    measured integer add and logic rates: one instruction per exact MAC is an
    upper bound for any CUDA-core Kulisch kernel), and exact GFLOP/s against the
    measured FP64 FMA flop rate (2 flops per fma), the pipe the page's kernel
    runs on.  Above 1.0 means the tensor-core residue path outruns that pipe's
    ceiling."""
    k = pipes["kinds"]
    int_peak = max(k["iadd"]["gops"], k["lop3"]["gops"])
    fp64 = 2.0 * k["dfma"]["gops"]
    return {"int32_issue": round(gflops / 2.0 / int_peak, 4),
            "int32_issue_peak_gops": int_peak,
            "fp64": round(gflops / fp64, 2), "fp64_peak_gflops": round(fp64, 1),
            "basis": "measured in this run (pipe_peaks): INT32 = max(iadd, lop3) instructions/s, "
                     "one per exact MAC; FP64 = 2 x dfma/s"}


def alu_peak_gops(sm_count, clock_mhz):
    """Nominal integer-ALU issue rate: SMs x 128 lanes x clock, one instruction
    per exact multiply-add counted as 2 ops (the same convention as 2MNK); only
    a fallback when no measured peak is at hand."""
    return 2.0 * sm_count * 128 * clock_mhz * 1e6 / 1e9


# ----------------------------------------------------------------------------- arms

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    A, B = make_inputs(0, args.workload)
    rows = max(1, args.cpu_rows // 4)
    cores = os.cpu_count() or 1
    g = np.random.default_rng(1234)

    def step():
        sel = np.sort(g.choice(M, size=rows, replace=False))
        oracle.gemm(np.ascontiguousarray(A[sel]), B, nthreads=cores)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = 2.0 * rows * N * K / dt / 1e9
    line = {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64",
            "data": "synthetic", "impl": "reference",
            # our arm's config (the oracle runs on the host cores: cpu_baseline)
            "config": workload_config(args.workload, {"parallelism": f"{world} independent replicas"
                                                      if world > 1 else "single GPU"}),
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                             "kind": "oracle",
                             "sample": f"each step: {rows} random rows of the 4096^3 problem"},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    import exact_sum_gemm_gb300 as dg
    from exact_sum_gemm_gb300 import _native
    lib = dg.library()

    nbatch = args.batch if args.op == "batched" else 1
    if args.op == "batched":                   # entries stacked along a leading axis
        from exact_sum_gemm_gb300 import workloads as wl
        A = wl.normal_f32((nbatch, M, K), rank_seed(rank), 0)
        B = wl.normal_f32((nbatch, N, K), rank_seed(rank), 1)
    else:
        A, B = make_inputs(rank_seed(rank), args.workload)
    a = torch.from_numpy(A).to(dev)
    b = torch.from_numpy(B).to(dev)
    c = torch.empty((nbatch, M, N) if nbatch > 1 else (M, N), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    if args.op == "batched":
        timed_call = lambda: dg.det_gemm_batched(a, b, out=c)
    elif args.op == "partial":
        digits = torch.empty((20, M, N), dtype=torch.int64, device=dev)
        timed_call = lambda: dg.det_gemm_partial(a, b, out=digits)
    else:
        timed_call = lambda: dg.det_gemm(a, b, out=c)

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(args.warmup):
        flush.zero_()
        timed_call()
    torch.cuda.synchronize(dev)

    props = torch.cuda.get_device_properties(dev)
    uuid = None
    try:
        uuid = "GPU-" + str(props.uuid)
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = lib.det_kernel_launches()
    barrier()
    torch.cuda.synchronize(dev)
    start.record(stream)
    for s in range(args.steps):
        flush.zero_()                  # L2 flush between steps, outside the step's events
        ev[s][0].record(stream)
        timed_call()
        ev[s][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    launches = lib.det_kernel_launches() - launches0
    clocks = sampler.stop()
    wall_ms = start.elapsed_time(end)
    kern_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    elapsed_ms = sum(kern_ms)          # the K steps' device time, flushes excluded
    if dist is not None:
        elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)
        wall_ms = max_over_ranks(wall_ms, dist, dev)
    ms_per_step = elapsed_ms / args.steps
    # stage breakdown: a separate pass with CUDA events around each stage
    stage_calls = min(args.steps, 5)
    lib.det_stage_timing(1)
    for _ in range(stage_calls):
        flush.zero_()
        timed_call()
    torch.cuda.synchronize(dev)
    lib.det_stage_timing(0)
    stages = stage_spans(_native.stage_timeline(), stage_calls)
    flops = 2.0 * M * N * K * nbatch
    value = flops * world / (ms_per_step * 1e-3) / 1e9

    extras = {"op": "det_gemm_partial"} if args.op == "partial" else {}
    if args.op == "batched":
        extras = {"op": "det_gemm_strided_batched", "batch": nbatch}
    if rank == 0 and not args.no_extras and args.op == "gemm":
        extras = measure_extras(args, dg, a, b, c, A, B, dev, stream)
    pipes = measure_pipe_peaks(lib, dev, uuid) if rank == 0 and not args.no_extras else None
    if rank == 0 and not args.no_extras and args.workload == "normal" and args.op == "gemm":
        del a, b, c
        torch.cuda.empty_cache()
        extras["workloads"] = measure_workloads(args, dev, pipes, with_cpu=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return 0

    peaks = measured_peaks()
    kern_avg = statistics.mean(kern_ms)
    # per det_gemm call: the time covered by a stage's records (a stage may
    # run once per row band, on several streams at once), so the stages need
    # not add up to the step
    stage_ms = {k: v[0] for k, v in stages.items()}
    # (the batched profiling mode has no per-entry roofline: its planes bound it)
    roofline = roofline_for(stage_ms, stages, props, peaks, lib, args.workload, pipes) \
        if args.op != "batched" else None
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "dtype_detail": DTYPE_DETAIL, "data": "synthetic",
        "config": workload_config(args.workload, {"parallelism": f"{world} independent replicas"
                                                  if world > 1 else "single GPU"}),
        "gpu_launches": int(launches),
        "timing": "sum of per-step CUDA-event intervals around det_gemm on its stream; the "
                  "256 MiB L2 flush between steps lies outside them",
        "wall_ms_per_step": round(wall_ms / args.steps, 4),
        "det_gemm_ms": round(kern_avg, 4),
        "stages_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "roofline": roofline,
        "pipe_fractions": pipe_fractions(value / world, pipes) if pipes else None,
        "pipe_peaks": pipes,
        "clocks": clocks,
    }
    line.update(extras)
    print(json.dumps(line), flush=True)
    return 0


def measure_extras(args, dg, a, b, c, A, B, dev, stream):
    import torch
    out = {}
    peaks = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    # ---- e2e: every step copies its inputs from pinned host memory and its
    # result back, inside the timed region.  Copies run on their own streams
    # (host->device, device->host) with double-buffered device tensors, so
    # step i+1's inputs travel while step i computes: a pipelined caller of
    # the public API.
    hA = torch.from_numpy(A).pin_memory()
    hB = torch.from_numpy(B).pin_memory()
    hC = [torch.empty((M, N), dtype=torch.float32).pin_memory() for _ in range(2)]
    dA = [a, torch.empty_like(a)]
    dB = [b, torch.empty_like(b)]
    dC = [c, torch.empty_like(c)]
    h2d = torch.cuda.Stream(dev)
    d2h = torch.cuda.Stream(dev)
    steps = max(4, min(args.steps, 10))

    def run(nsteps):
        gemm_done = [None, None]
        for i in range(nsteps):
            j = i % 2
            with torch.cuda.stream(h2d):
                if gemm_done[j] is not None:
                    h2d.wait_event(gemm_done[j])        # buffer j free again
                dA[j].copy_(hA, non_blocking=True)
                dB[j].copy_(hB, non_blocking=True)
                copied = torch.cuda.Event()
                copied.record(h2d)
            stream.wait_event(copied)
            dg.det_gemm(dA[j], dB[j], out=dC[j])
            done = torch.cuda.Event()
            done.record(stream)
            gemm_done[j] = done
            with torch.cuda.stream(d2h):
                d2h.wait_event(done)
                hC[j].copy_(dC[j], non_blocking=True)

    run(2)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d.wait_event(e0)
    run(steps)
    d2h.wait_stream(stream)
    d2h.wait_stream(h2d)
    e1.record(d2h)
    torch.cuda.synchronize(dev)
    t = e0.elapsed_time(e1) / steps
    out["e2e"] = {"value": round(2.0 * M * N * K / (t * 1e-3) / 1e9, 3), "unit": UNIT,
                  "h2d_bytes_per_step": int(A.nbytes + B.nbytes),
                  "d2h_bytes_per_step": int(hC[0].nbytes), "ms_per_step": round(t, 4),
                  "pipelining": "double-buffered; copies on separate streams overlap the GEMM"}
    del dA[1], dB[1], dC[1]
    # ---- the same det_gemm captured once in a CUDA graph and replayed: the
    # launches of a call go to the GPU as one graph (flush outside the events)
    out_g = torch.empty_like(c)
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        dg.det_gemm(a, b, out=out_g)
    stream.wait_stream(side)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dg.det_gemm(a, b, out=out_g)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(3):
        flush.zero_()
        graph.replay()
    torch.cuda.synchronize(dev)
    g_ms = []
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        g_ms.append(e0.elapsed_time(e1))
    tg = statistics.mean(g_ms)
    out["graph_replay"] = {
        "value": round(2.0 * M * N * K / (tg * 1e-3) / 1e9, 3), "unit": UNIT,
        "ms_per_step": round(tg, 4),
        "equal_to_eager": bool(torch.equal(out_g.view(torch.int32), c.view(torch.int32)))}
    del graph, out_g, flush
    # ---- sharded: 2-way K split through partial / combine / finalize
    full_bits = c.clone()
    cuts = [(0, K // 2), (K // 2, K)]
    P = [torch.empty((20, M, N), dtype=torch.int64, device=dev) for _ in cuts]
    acc = torch.empty((20, M, N), dtype=torch.int64, device=dev)
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    times = {"partial": [], "combine": [], "finalize": []}
    for rep in range(3):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        evs[0].record(stream)
        for (k0, k1), p in zip(cuts, P):
            dg.det_gemm_partial(a[:, k0:k1], b[:, k0:k1], out=p)
        evs[1].record(stream)
        dg.det_combine(P, out=acc)
        evs[2].record(stream)
        dg.det_finalize(acc, out=y)
        evs[3].record(stream)
        torch.cuda.synchronize(dev)
        if rep > 0:
            times["partial"].append(evs[0].elapsed_time(evs[1]))
            times["combine"].append(evs[1].elapsed_time(evs[2]))
            times["finalize"].append(evs[2].elapsed_time(evs[3]))
    equal = bool(torch.equal(y.view(torch.int32), full_bits.view(torch.int32)))
    tc = statistics.mean(times["combine"])
    tf = statistics.mean(times["finalize"])
    tp = statistics.mean(times["partial"])
    comb_bytes = 3 * 20 * 8 * M * N            # read 2 partials, write 1
    fin_bytes = (19 * 8 + 4) * M * N           # read 18 digits + non-finite plane, write fp32
    out["sharded"] = {
        "equal_to_full_k": equal, "shards": 2,
        "ms": {"partials": round(tp, 3), "combine": round(tc, 3), "finalize": round(tf, 3)},
        "value": round(2.0 * M * N * K / ((tp + tc + tf) * 1e-3) / 1e9, 3), "unit": UNIT,
        "combine_roofline": {"bound": "hbm", "achieved": round(comb_bytes / (tc * 1e-3) / 1e9, 1),
                             "peak": hbm, "unit": "GB/s",
                             "frac": round(comb_bytes / (tc * 1e-3) / 1e9 / hbm, 4),
                             "algorithmic_bytes": comb_bytes},
        "finalize_roofline": {"bound": "hbm", "achieved": round(fin_bytes / (tf * 1e-3) / 1e9, 1),
                              "peak": hbm, "unit": "GB/s",
                              "frac": round(fin_bytes / (tf * 1e-3) / 1e9 / hbm, 4),
                              "algorithmic_bytes": fin_bytes},
    }
    del P, acc
    torch.cuda.empty_cache()
    # ---- CPU oracle baseline (bounded sample)
    out["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_rows)
    return out


def oracle_time(fn, macs, cores, sample):
    """The CPU oracle as it stands, timed once on the host cores."""
    t0 = time.perf_counter()
    fn()
    dt = time.perf_counter() - t0
    return {"value": round(2.0 * macs / dt / 1e9, 4), "unit": UNIT, "cores": cores,
            "kind": "oracle", "sample": f"{sample}; {dt:.2f} s wall on {cores} threads",
            "seconds": round(dt, 2)}


def measure_workloads(args, dev, pipes=None, with_cpu=True):
    """Every workload configuration, timed on one GPU with inputs resident in
    HBM: CUDA events on the current stream around `steps` calls after `warmup`
    calls (no L2 flush: the small problems fit in L2 by design).  Exact GFLOP/s
    counts 2MNK per GEMM.  Beside each, the exact work rate against the
    measured INT32 issue and FP64 peaks, and the CPU oracle timed on the host
    cores (full problems, or a stated sample)."""
    import torch
    import exact_sum_gemm_gb300 as dg
    from exact_sum_gemm_gb300 import workloads as wl
    torch.cuda.set_device(dev)
    steps, warm = max(2, min(args.steps, 5)), max(1, min(args.warmup, 2))
    cores = os.cpu_count() or 1
    if with_cpu:
        import oracle
        oracle.build()
    out = {}

    def timed(fn, n=steps):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / n

    def entry(name, desc, ms, flops, cpu=None, **extra):
        g = flops / (ms * 1e-3) / 1e9
        e = {"workload": desc, "ms": round(ms, 4), "exact_gflops": round(g, 2)}
        if pipes:
            pf = pipe_fractions(g, pipes)
            e["vs_int32_issue"] = pf["int32_issue"]
            e["vs_fp64"] = pf["fp64"]
        if cpu is not None:
            e["cpu_baseline"] = cpu
        e.update(extra)
        out[name] = e
        if args.configs:
            print(json.dumps({"config": name, **e, "data": "synthetic"}), flush=True)

    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
    # 64^3 f32 N(0,1): det_gemm, and 16 equal K-shards through partial/combine/finalize
    A1, B1 = wl.normal_f32((64, 64), 0, 0), wl.normal_f32((64, 64), 0, 1)
    a, b = f32(A1), f32(B1)
    cpu = oracle_time(lambda: oracle.gemm(A1, B1, nthreads=cores), 64 ** 3, cores,
                      "the full 64^3 problem") if with_cpu else None
    entry("c1_det_gemm", "det_gemm f32 64x64x64 N(0,1), seed 0",
          timed(lambda: dg.det_gemm(a, b)), 2.0 * 64 ** 3, cpu)
    cuts = wl.equal_cuts(64, 16)
    entry("c1_shards16", "det_gemm_partial x16 + det_combine + det_finalize, same problem",
          timed(lambda: dg.det_gemm_sharded(a, b, cuts)), 2.0 * 64 ** 3)
    # bf16 512x512x4096, exponents U{-60..60}, cancelling column pairs; 8 random K-shards
    A2, B2, _ = wl.bf16_wide_with_cancellation(512, 512, 4096, 1)
    ab, bb = wl.to_torch_bf16(A2, dev), wl.to_torch_bf16(B2, dev)
    fl = 2.0 * 512 * 512 * 4096
    cpu = oracle_time(lambda: oracle.gemm(A2, B2, dtype="bf16", nthreads=cores), fl / 2, cores,
                      "the full 512x512x4096 problem") if with_cpu else None
    entry("c2_det_gemm", "det_gemm bf16 512x512x4096, exponents U{-60..60}, cancelling pairs, "
          "seed 1", timed(lambda: dg.det_gemm(ab, bb)), fl, cpu)
    rcuts = wl.kshard_cuts(4096, 8, 1)
    entry("c2_shards8", "det_gemm_partial x8 (random cuts) + combine + finalize, same problem",
          timed(lambda: dg.det_gemm_sharded(ab, bb, rcuts)), fl)
    # DetLinear 4096 -> 4096 on a 2048 x 4096 batch: forward, dgrad, wgrad
    x_np, w_np = wl.detlinear_inputs()
    x, w = f32(x_np), f32(w_np)
    y = dg.det_linear_forward(x, w)
    dy = (y * 2.0 ** -22).contiguous()
    fl = 2.0 * 2048 * 4096 * 4096
    cpu_f = cpu_d = cpu_w = None
    if with_cpu:
        cpu_f = oracle_time(lambda: oracle.gemm(x_np, w_np, nthreads=cores), fl / 2, cores,
                            "the full forward GEMM (2048x4096x4096)")
        # the oracle's time does not depend on which upstream gradient it is
        # given: a generator draw of the same scale stands in for dy
        dy_np = wl.normal_f32((256, 4096), 2, 5, scale_pow2=-22)
        w_t = np.ascontiguousarray(w_np.T)
        cpu_d = oracle_time(lambda: oracle.gemm(dy_np, w_t, nthreads=cores), 256 * 4096 * 4096,
                            cores, "256 of the 2048 rows of dgrad (each row costs the same)")
        dyt = wl.normal_f32((256, 2048), 2, 6, scale_pow2=-22)
        x_t = np.ascontiguousarray(x_np.T)
        cpu_w = oracle_time(lambda: oracle.gemm(dyt, x_t, nthreads=cores), 256 * 4096 * 2048,
                            cores, "256 of the 4096 rows of wgrad (each row costs the same)")
    entry("c3_forward", "DetLinear 4096->4096 forward, x 2048x4096 N(0,1), W N(0,1)/64, seed 2",
          timed(lambda: dg.det_linear_forward(x, w)), fl, cpu_f)
    entry("c3_dgrad", "DetLinear dgrad (dy = 2y/numel)", timed(lambda: dg.det_linear_dgrad(dy, w)),
          fl, cpu_d)
    entry("c3_wgrad", "DetLinear wgrad", timed(lambda: dg.det_linear_wgrad(dy, x)), fl, cpu_w)
    del x, w, y, dy
    # f32 256x256, K = 2^19, |x| = 2^U[-100,100]
    KL = 1 << 19
    A4, B4 = wl.loguniform_f32((256, KL), 3, 0), wl.loguniform_f32((256, KL), 3, 1)
    a4, b4 = f32(A4), f32(B4)
    cpu = oracle_time(lambda: oracle.gemm(A4, B4, nthreads=cores), 256 * 256 * KL, cores,
                      "the full 256x256x524288 problem") if with_cpu else None
    entry("c4_det_gemm", "det_gemm f32 256x256x524288, |x| = 2^U[-100,100], seed 3",
          timed(lambda: dg.det_gemm(a4, b4), n=2), 2.0 * 256 * 256 * KL, cpu)
    del a4, b4, A4, B4
    # the headline shape with wide exponents: |x| = 2^U[-40,40]
    Aw = wl.loguniform_f32((4096, 4096), 0, 0, lo=-40, hi=40)
    Bw = wl.loguniform_f32((4096, 4096), 0, 1, lo=-40, hi=40)
    aw, bw = f32(Aw), f32(Bw)
    cpu = oracle_time(lambda: oracle.gemm(np.ascontiguousarray(Aw[::64]), Bw, nthreads=cores),
                      64 * 4096 * 4096, cores, "64 evenly spaced rows of the 4096^3 problem") \
        if with_cpu else None
    entry("wide_4096", "det_gemm f32 4096^3, |x| = 2^U[-40,40], seed 0",
          timed(lambda: dg.det_gemm(aw, bw), n=3), 2.0 * 4096 ** 3, cpu)
    del aw, bw, Aw, Bw
    # the headline shape with a few wide rows: N(0,1), rows 1024..1151 of A
    # with |x| = 2^U[-40,40] (their tiles go to the wide path, the rest stay
    # on the narrow one)
    Am = wl.normal_f32((4096, 4096), 0, 0)
    Am[1024:1152] = wl.loguniform_f32((128, 4096), 5, 0, lo=-40, hi=40)
    Bm = wl.normal_f32((4096, 4096), 0, 1)
    am, bm = f32(Am), f32(Bm)
    cpu = oracle_time(lambda: oracle.gemm(np.ascontiguousarray(Am[1024:1088]), Bm, nthreads=cores),
                      64 * 4096 * 4096, cores, "64 of the wide rows of the 4096^3 problem") \
        if with_cpu else None
    entry("mixed_4096", "det_gemm f32 4096^3, A,B N(0,1) seed 0 with rows 1024..1151 of A "
          "|x| = 2^U[-40,40] (seed 5)", timed(lambda: dg.det_gemm(am, bm), n=5),
          2.0 * 4096 ** 3, cpu)
    del am, bm, Am, Bm
    # one training step of the 1024 -> 4096 -> 1024 MLP, batch 256 (targets
    # from the teacher through det_gemm, forward, backward, SGD update)
    relu = lambda t: torch.clamp_min(t, 0.0)
    w1, w2 = wl.mlp_init(stream=0)
    t1, t2 = wl.mlp_init(stream=1)
    t1d, t2d = f32(t1), f32(t2)
    x5 = wl.mlp_batch(0)
    xb = f32(x5)
    lr = torch.tensor(1e-2, dtype=torch.float32, device=dev)
    cpu = None
    if with_cpu:
        h_np = np.ascontiguousarray(x5[:32])
        cpu = oracle_time(lambda: oracle.gemm(h_np, t1, nthreads=cores), 32 * 4096 * 1024, cores,
                          "32 of the 256 rows of the step's first GEMM (each of the seven GEMMs "
                          "is 256x4096x1024 or its transpose, so the rate carries over)")
    for shards in (1, 4):
        l1 = dg.DetLinear(1024, 4096, device=dev, k_shards=shards, weight=torch.from_numpy(w1))
        l2 = dg.DetLinear(4096, 1024, device=dev, k_shards=shards, weight=torch.from_numpy(w2))

        def step():
            with torch.no_grad():
                target = dg.det_gemm(relu(dg.det_gemm(xb, t1d)), t2d)
            loss = (l2(relu(l1(xb))) - target).square().mean()
            for q in (l1.weight, l2.weight):
                q.grad = None
            loss.backward()
            with torch.no_grad():
                for q in (l1.weight, l2.weight):
                    q.sub_(q.grad * lr)
        # 2 teacher + 2 forward + 1 dgrad + 2 wgrad GEMMs of 256 x 1024 x 4096
        entry(f"c5_step_shards{shards}", f"MLP 1024->4096->1024 training step, batch 256, "
              f"k_shards={shards}, seed 7", timed(step), 7 * 2.0 * 256 * 1024 * 4096,
              cpu if shards == 1 else None)
    del l1, l2, t1d, t2d, xb
    # strided batch: 64 attention-like heads of 128 x 128 x 4096, one pipeline
    # against the same entries enqueued one after another
    lib = dg.library()
    nb, mb, kb = 64, 128, 4096
    Ab, Bb = wl.normal_f32((nb, mb, kb), 61, 0), wl.normal_f32((nb, mb, kb), 61, 1)
    xb3, wb3 = f32(Ab), f32(Bb)
    outb = torch.empty((nb, mb, mb), dtype=torch.float32, device=dev)
    call = lambda: dg.det_gemm_batched(xb3, wb3, out=outb)
    fl = 2.0 * nb * mb * mb * kb

    def launches(fn):
        torch.cuda.synchronize(dev)
        n0 = lib.det_kernel_launches()
        fn()
        torch.cuda.synchronize(dev)
        return int(lib.det_kernel_launches() - n0)
    n_pipe, t_pipe = launches(call), timed(call)
    prev = lib.det_set_batched_pipeline(0)
    n_loop, t_loop = launches(call), timed(call)
    lib.det_set_batched_pipeline(prev)
    cpu = oracle_time(lambda: oracle.gemm(Ab[0], Bb[0], nthreads=cores), mb * mb * kb, cores,
                      "one of the 64 entries (each costs the same)") if with_cpu else None
    entry("batched_64x128x128x4096", "det_gemm_strided_batched f32, 64 entries of 128x128x4096 "
          "N(0,1), seed 61", t_pipe, fl, cpu, launches=n_pipe,
          entry_by_entry={"ms": round(t_loop, 4), "exact_gflops": round(fl / (t_loop * 1e-3) / 1e9, 2),
                          "launches": n_loop},
          speedup=round(t_loop / t_pipe, 2))
    return out


def run_configs(args):
    """Each workload configuration timed on one GPU (one JSON line each)."""
    import torch
    measure_workloads(args, torch.device("cuda", 0), None, with_cpu=False)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.configs:
        return run_configs(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
