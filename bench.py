#!/usr/bin/env python
"""Benchmark: ring all-reduce of N virtual ranks on one GB300.

Default workload: 8 ranks x 64 Mi fp32 elements (256 MiB per rank), op avg,
per-rank seeded normal(0, 1e-3) gradients. One step = one ra_allreduce call
(one fused kernel launch) over inputs already resident in HBM. The metric is
the all-reduce algorithm bandwidth S/t (S = bytes per rank), aggregated over
GPUs when run as replicas under torchrun; the roofline block gives the HBM
fraction of the algorithmic traffic 2*N*S per launch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
    python bench.py --sweep OUT.jsonl      # message-size sweep, one line per (N, size, call)
    python bench.py --overlap              # bucketed all-reduce beside a synthetic backward pass
    python bench.py --roofs                # read/write stream rates the kernels are compared against
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

from ring_all_reduce_02_gb300 import inputs  # noqa: E402

METRIC = "all-reduce algorithm GB/s and % of HBM roofline vs message size, N=8 ranks, 1 GPU"
DEFAULT_WORKLOAD = "ar_n8_f32_avg_64m"
GB = 1e9


# ---------------------------------------------------------------------------
# environment: ranks, peaks, clocks
# ---------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []  # (t, sm_mhz, max_mhz, reasons[list])
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm, mx = float(f[1]), float(f[2])
            except ValueError:
                continue
            reasons = [n for n, v in zip(names, f[5:9]) if v.lower() == "active"]
            self.samples.append((time.time(), sm, mx, reasons))

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
        inside = [s for s in self.samples if t0 - 0.15 <= s[0] <= t1 + 0.15]
        used = inside if len(inside) >= 2 else self.samples
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({r for s in used for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in used), "sm_max_mhz": max(s[2] for s in used),
                "reasons": reasons, "samples": len(used), "in_timed_region": len(inside)}


def max_over_ranks(ms: float, world: int, device: str) -> float:
    """The slowest rank's time: the job is done when every replica is done."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(bytes_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job algorithm bandwidth: every replica reduces bytes_per_rank per step."""
    return world * bytes_per_rank / (ms_per_step * 1e-3) / GB


# the sources that define the fused all-reduce kernel's code
AR_KERNEL_SOURCES = ("ra_kernels.cuh", "ra_ops.cuh", "ra_plan.h")


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ring_all_reduce_02_gb300", "csrc")
    for f in AR_KERNEL_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel source."""
    p = os.path.join(ROOT, "profiles", f"ar_fused_kernel__{workload}.txt")
    if not os.path.exists(p):
        return None
    kv = {}
    with open(p) as f:
        for ln in f:
            if ":" in ln:
                k, v = ln.split(":", 1)
                kv[k.strip()] = v.strip()
    if kv.get("kernel_source_sha256_16") != kernel_source_sha():
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# the CPU oracle as a baseline (bounded sample of the same workload)
# ---------------------------------------------------------------------------
def host_cpu() -> dict:
    """The host the CPU baseline ran on: logical CPUs (nproc) and the lscpu model name."""
    try:
        nproc = len(os.sched_getaffinity(0))
    except AttributeError:
        nproc = os.cpu_count() or 1
    model = vendor = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            k, _, v = ln.partition(":")
            if k.strip() == "Model name" and model is None:
                model = v.strip()
            elif k.strip() == "Vendor ID" and vendor is None:
                vendor = v.strip()
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None and os.path.exists("/proc/cpuinfo"):
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    model = ln.split(":", 1)[1].strip()
                    break
    return {"nproc": nproc, "cpu_model": model or "unknown", "cpu_vendor": vendor or "unknown"}


def oracle_rate(n, length, dtype, op, dist, target_s: float, max_len: int, repeat: bool = False):
    """Time the oracle on a sample of the workload sized to about target_s; returns (GB/s, sample_len, secs,
    runs). A sample capped at the whole workload is run again (repeat=True) until about target_s has passed."""
    import oracle

    oracle.build()
    probe = min(max_len, 1 << 20)
    xs = inputs.rank_buffers(n, probe, dtype, dist)
    t = time.perf_counter()
    oracle.allreduce(xs, op, dtype)
    dt = max(time.perf_counter() - t, 1e-4)
    sample = int(min(max_len, max(4096 * n, probe * target_s / dt)))
    xs = inputs.rank_buffers(n, sample, dtype, dist)
    runs, total = 0, 0.0
    while runs == 0 or (repeat and total < target_s and runs < 100):
        t = time.perf_counter()
        oracle.allreduce(xs, op, dtype)
        total += time.perf_counter() - t
        runs += 1
    s_bytes = sample * inputs.ELEM_SIZE[dtype]
    return s_bytes * runs / total / GB, sample, total, runs


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    n, length, dtype, op, dist = inputs.WORKLOADS[args.workload]
    import oracle

    oracle.build()
    # size each step so warm-up + timed steps take about a minute in total
    _, sample, _, _ = oracle_rate(n, length, dtype, op, dist,
                                  target_s=min(5.0, 60.0 / max(1, args.steps + args.warmup)), max_len=length)
    xs = inputs.rank_buffers(n, sample, dtype, dist)
    for _ in range(args.warmup):
        oracle.allreduce(xs, op, dtype)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.allreduce(xs, op, dtype)
        times.append(time.perf_counter() - t)
    total = sum(times)
    s_bytes = sample * inputs.ELEM_SIZE[dtype]
    value = s_bytes * args.steps / total / GB
    cores = min(n, os.cpu_count() or 1)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
        "config": config_block(args.workload),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} ranks x {sample} {dtype} elements per step (the workload is {length})",
                         **host_cpu()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_block(workload: str):
    n, length, dtype, op, dist = inputs.WORKLOADS[workload]
    s_bytes = length * inputs.ELEM_SIZE[dtype]
    return {"workload": workload, "nranks": n, "count": length, "dtype": dtype, "op": op,
            "bytes_per_rank": s_bytes, "inputs": f"seeded {dist[0]}{tuple(dist[1:])}, seed = rank",
            "l2": f"inputs larger than L2 ({2 * n * s_bytes / GB:.1f} GB touched per step vs ~0.13 GB L2)",
            "parallelism": "replicas (one N-rank instance per GPU)"}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    from ring_all_reduce_02_gb300 import build, ra

    build.build()
    ra.lib()
    dev = torch.cuda.current_device()
    n, length, dtype, op, dist_spec = inputs.WORKLOADS[args.workload]
    es = inputs.ELEM_SIZE[dtype]
    s_bytes = length * es
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "i32": torch.int32}[dtype]

    host = inputs.rank_buffers(n, length, dtype, dist_spec)
    pinned_in, sends = [], []
    for x in host:
        t = torch.from_numpy(x.view(np.int16) if dtype == "bf16" else x)
        p = t.pin_memory()
        pinned_in.append(p.view(tdt) if dtype == "bf16" else p)
        sends.append(pinned_in[-1].to(f"cuda:{dev}"))
    del host
    recvs = [torch.empty_like(s) for s in sends]
    stream = torch.cuda.current_stream()

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            torch.cuda.synchronize()

    for _ in range(args.warmup):
        ra.ra_allreduce(sends, recvs, op, stream=stream)
    sampler = ClockSampler(dev).start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    t_wall0 = time.time()
    for k in range(args.steps):
        starts[k].record(stream)
        ra.ra_allreduce(sends, recvs, op, stream=stream)
        ends[k].record(stream)
    barrier()
    t_wall1 = time.time()
    launches = args.steps  # one fused kernel per call
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]  # ms, per launch
    total_ms = max_over_ranks(starts[0].elapsed_time(ends[-1]), world, f"cuda:{dev}")
    time.sleep(0.2)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)

    ms_per_step = total_ms / args.steps
    value = job_value(s_bytes, world, ms_per_step)
    avg_launch_ms = sum(per) / len(per)
    peak, peak_kind = measured_peaks()
    achieved = 2 * n * s_bytes / (avg_launch_ms * 1e-3) / GB
    traffic = profiled_traffic(args.workload)

    # End to end through the C ABI with host buffers: every step the call reads all N ranks' inputs
    # from pinned host memory and writes all N results to pinned host memory (the kernel moves the
    # bytes over the host link itself: N*S host->device and N*S device->host per step). For
    # comparison, the same step staged through device buffers with copy-engine transfers.
    e2e_steps = max(3, min(args.steps, 20))
    pinned_out = [torch.empty(r.shape, dtype=r.dtype, pin_memory=True) for r in recvs]
    dt_code, op_code = ra.DTYPE_CODES[dtype], ra.OP_CODES[op]
    host_in = [p.data_ptr() for p in pinned_in]
    host_out = [p.data_ptr() for p in pinned_out]

    def host_step():
        rc = ra.call("ra_allreduce", host_in, host_out, length, dt_code, op_code, n, stream.cuda_stream)
        if rc:
            raise ra.RaError(rc, "ra_allreduce (host buffers)")

    def staged_step():
        for p, s in zip(pinned_in, sends):
            s.copy_(p, non_blocking=True)
        ra.ra_allreduce(sends, recvs, op, stream=stream)
        for p, r in zip(pinned_out, recvs):
            p.copy_(r, non_blocking=True)

    def time_steps(step):
        for _ in range(2):
            step()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            step()
        e1.record(stream)
        barrier()
        return max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, f"cuda:{dev}")

    e2e_ms = time_steps(host_step)
    e2e_value = job_value(s_bytes, world, e2e_ms)
    staged_ms = time_steps(staged_step)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, sample, secs, runs = oracle_rate(n, length, dtype, op, dist_spec, target_s=10.0, max_len=length,
                                               repeat=True)
        cpu = {"value": round(rate, 4), "unit": "GB/s", "cores": min(n, os.cpu_count() or 1), "kind": "oracle",
               "sample": f"{n} ranks x {sample} {dtype} elements, {runs} run(s) ({secs:.1f} s, one thread per rank)",
               **host_cpu()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
            "config": config_block(args.workload),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "kernel": "ar_fused_kernel", "algorithmic_bytes_per_launch": 2 * n * s_bytes,
                         "peak_source": f"{peak_kind} hbm_gbs (copy, burst)",
                         "launch_ms": {"mean": round(avg_launch_ms, 5), "min": round(min(per), 5),
                                       "median": round(statistics.median(per), 5)}},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 3), "unit": "GB/s", "h2d_bytes_per_step": n * s_bytes,
                    "d2h_bytes_per_step": n * s_bytes, "ms_per_step": round(e2e_ms, 4),
                    "path": "ra_allreduce on pinned host buffers (kernel reads and writes host memory)",
                    "staged_ms_per_step": round(staged_ms, 4),
                    "staged_value": round(job_value(s_bytes, world, staged_ms), 3)},
            "gpu_launches": launches,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# message-size sweep (not the headline line): AR / RS / AG timed separately
# ---------------------------------------------------------------------------
def run_sweep(args):
    import torch

    from ring_all_reduce_02_gb300 import build, ra

    build.build()
    torch.cuda.set_device(0)
    peak, peak_kind = measured_peaks()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(int(2 * l2), dtype=torch.uint8, device="cuda")
    # read after the flush to write its dirty lines back: the "clean" timing starts from an L2
    # that holds only clean lines of unrelated data
    evict = torch.ones(int(2 * l2) // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    out = open(args.sweep, "w")
    for (n, length, dtype, op, dist_spec) in inputs.size_sweep():
        if args.sweep_max and length > args.sweep_max:
            continue
        es = inputs.ELEM_SIZE[dtype]
        s_bytes = length * es
        g = torch.Generator(device="cuda")
        g.manual_seed(0)
        sends = [torch.empty(length, dtype=torch.float32, device="cuda").uniform_(-1, 1, generator=g) for _ in range(n)]
        recvs = [torch.empty_like(s) for s in sends]
        bounds = [ra.ra_chunk_range(length, n, c) for c in range(n)]
        shards = [torch.empty(e - b, dtype=torch.float32, device="cuda") for b, e in bounds]
        calls = {
            "allreduce": (lambda: ra.ra_allreduce(sends, recvs, op, stream=stream), 2 * n * s_bytes),
            "reduce_scatter": (lambda: ra.ra_reduce_scatter(sends, shards, op, stream=stream), (n + 1) * s_bytes),
            "allgather": (lambda: ra.ra_allgather(shards, recvs, stream=stream), (n + 1) * s_bytes),
        }
        for name, (fn, hbm_bytes) in calls.items():
            resident = hbm_bytes < l2
            for _ in range(5):
                fn()
            reps = 20

            def timed_reps(clean):
                times = []
                for _ in range(reps):
                    if not resident:
                        flush.zero_()
                        if clean:
                            torch.amax(evict)
                    # keep the GPU busy until the launch and both events are queued, so that the
                    # interval holds the kernel alone and none of the host's call overhead
                    torch.cuda._sleep(200_000)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    fn()
                    b.record(stream)
                    torch.cuda.synchronize()
                    times.append(a.elapsed_time(b) * 1e-3)
                return times

            times = timed_reps(False)
            rec = {"call": name, "nranks": n, "bytes_per_rank": s_bytes, "count": length,
                   "median_us": round(1e6 * statistics.median(times), 3), "min_us": round(1e6 * min(times), 3),
                   "algbw_GBps": round(s_bytes / statistics.median(times) / GB, 3),
                   "hbm_GBps": round(hbm_bytes / statistics.median(times) / GB, 1),
                   "hbm_frac": None if resident else round(hbm_bytes / statistics.median(times) / GB / peak, 4),
                   "l2_resident": resident, "peak": f"{peak} ({peak_kind})"}
            if not resident:
                clean = statistics.median(timed_reps(True))
                rec["clean_median_us"] = round(1e6 * clean, 3)
                rec["clean_hbm_frac"] = round(hbm_bytes / clean / GB / peak, 4)
            if resident:
                # warm, back-to-back launches captured in one CUDA graph: launch cost amortised
                gs = torch.cuda.Stream()
                gs.wait_stream(stream)
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.stream(gs):
                    fn_g = {"allreduce": lambda: ra.ra_allreduce(sends, recvs, op, stream=gs),
                            "reduce_scatter": lambda: ra.ra_reduce_scatter(sends, shards, op, stream=gs),
                            "allgather": lambda: ra.ra_allgather(shards, recvs, stream=gs)}[name]
                    fn_g()
                    torch.cuda.synchronize()
                    with torch.cuda.graph(graph, stream=gs):
                        for _ in range(100):
                            fn_g()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                graph.replay()
                torch.cuda.synchronize()
                a.record(stream)
                graph.replay()
                b.record(stream)
                torch.cuda.synchronize()
                rec["graph_us_per_call"] = round(1e3 * a.elapsed_time(b) / 100, 3)
            out.write(json.dumps(rec) + "\n")
            out.flush()
            print(json.dumps(rec), flush=True)
        del sends, recvs, shards
        torch.cuda.empty_cache()
    out.close()
    return 0


# ---------------------------------------------------------------------------
# one call of the library timed alone on a workload's buffers (not the headline):
# per-kernel rooflines and the command that ncu captures of each kernel run
# ---------------------------------------------------------------------------
CALLS = {  # name: (kernel, algorithmic bytes per launch as a multiple of S, the bytes per rank)
    "allreduce": ("ar_fused_kernel", lambda n: 2 * n),
    "reduce_scatter": ("rs_fused_kernel", lambda n: n + 1),
    "allgather": ("ag_tma_store_kernel (N <= 4, N = 8) or ag_tma_flat_kernel", lambda n: n + 1),
    "allreduce_bulk": ("ar_bulk_kernel", lambda n: 2 * n),
    "allreduce_fp32acc": ("ar_fused_kernel (fp32 partials)", lambda n: 2 * n),
    "allreduce_tree": ("ordered_kernel", lambda n: 2 * n),
    "allreduce_rabenseifner": ("ordered_kernel", lambda n: 2 * n),
    # the literal schedule: per reduce-scatter step 3 S (read the incoming partial and the own
    # chunk, write the sum), per all-gather step 2 S, over N-1 steps each
    "allreduce_ringsteps": ("ring_rs_step_kernel + ring_ag_step_kernel", lambda n: 5 * (n - 1)),
}


def run_call(args):
    import torch

    from ring_all_reduce_02_gb300 import build, ra

    build.build()
    torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    n, length, dtype, op, _ = inputs.WORKLOADS[args.workload]
    workload = args.workload
    if args.case:  # an explicit case instead of a named workload: N,COUNT,DTYPE,OP
        n_s, count_s, dtype, op = args.case.split(",")
        n, length = int(n_s), int(count_s)
        workload = f"case_n{n}_{dtype}_{op}_{length}"
    es = inputs.ELEM_SIZE[dtype]
    s_bytes = length * es
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "i32": torch.int32}[dtype]
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    sends = [torch.empty(length, dtype=torch.float32, device="cuda").normal_(generator=g).to(tdt) for _ in range(n)]
    recvs = [torch.empty_like(x) for x in sends]
    bounds = [ra.ra_chunk_range(length, n, c) for c in range(n)]
    shards = [x[b:e].clone() for x, (b, e) in zip(sends, bounds)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    name = args.call
    fn = {
        "allreduce": lambda: ra.ra_allreduce(sends, recvs, op, stream=stream),
        "reduce_scatter": lambda: ra.ra_reduce_scatter(sends, shards, op, stream=stream),
        "allgather": lambda: ra.ra_allgather(shards, recvs, stream=stream),
        "allreduce_bulk": lambda: ra.ra_allreduce_ex(sends, recvs, op, engine="bulk", status=status, stream=stream),
        "allreduce_fp32acc": lambda: ra.ra_allreduce_ex(sends, recvs, op, accum="fp32", stream=stream),
        "allreduce_tree": lambda: ra.ra_allreduce_ex(sends, recvs, op, order="tree", stream=stream),
        "allreduce_rabenseifner": lambda: ra.ra_allreduce_ex(sends, recvs, op, order="rabenseifner", stream=stream),
        "allreduce_ringsteps": lambda: ra.ra_allreduce_ringsteps(sends, recvs, op, stream=stream),
    }[name]
    kernel, mult = CALLS[name]
    hbm_bytes = mult(n) * s_bytes
    for _ in range(args.warmup):
        fn()
    sampler = ClockSampler(dev).start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for k in range(args.steps):
        starts[k].record(stream)
        fn()
        ends[k].record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    time.sleep(0.2)
    sampler.stop()
    per = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    mean_ms = sum(per) / len(per)
    peak, peak_kind = measured_peaks()
    achieved = hbm_bytes / (mean_ms * 1e-3) / GB
    print(json.dumps({
        "mode": "call", "call": name, "kernel": kernel, "workload": workload, "nranks": n, "count": length,
        "dtype": dtype, "op": op, "steps": args.steps, "warmup": args.warmup,
        "inputs": "seeded normal(0, 1) drawn on the device",
        "l2": f"{hbm_bytes / GB:.2f} GB moved per launch vs ~0.13 GB L2",
        "algorithmic_bytes_per_launch": hbm_bytes,
        "launch_ms": {"mean": round(mean_ms, 5), "min": round(min(per), 5), "median": round(statistics.median(per), 5)},
        "achieved_GBps": round(achieved, 1), "peak": peak, "peak_source": f"{peak_kind} hbm_gbs (copy, burst)",
        "frac": round(achieved / peak, 4), "status": int(status.item()),
        "algbw_GBps": round(s_bytes / (mean_ms * 1e-3) / GB, 3),
        "clocks": sampler.summary(t_wall0, t_wall1)}), flush=True)
    return 0 if status.item() == 0 else 1


# ---------------------------------------------------------------------------
# bucketed all-reduce overlapped with a synthetic backward pass (not the headline)
# ---------------------------------------------------------------------------
def run_overlap(args):
    """DDP-style 25 MB buckets of the 8-rank bf16 GPT-2-medium gradient bucket, each all-reduced on a
    communication stream as soon as a synthetic backward GEMM on the compute stream has produced it.
    Reports compute-only, all-reduce-only and overlapped times for several SM budgets."""
    import torch

    from ring_all_reduce_02_gb300 import build, ra

    build.build()
    torch.cuda.set_device(0)
    n, length, dtype, op, _ = inputs.WORKLOADS["ar_n8_bf16_avg_gpt2m"]
    counts = [int(np.prod(s)) for _, s in inputs.gpt2_medium_param_shapes()]
    plan = ra.ra_bucket_plan(counts, 25 * 1000 * 1000, 2)
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    sends = [(torch.randn(length, device="cuda", generator=g) * 0.01).to(torch.bfloat16) for _ in range(n)]
    recvs = [torch.empty_like(s) for s in sends]
    # synthetic backward: bucket b's weight gradient costs 2 * count_b * tokens flops (one bf16 GEMM
    # [count_b/1024 x tokens] @ [tokens x 1024]), produced in the order the buckets become ready
    tokens = args.overlap_tokens
    gy = torch.randn(tokens, 1024, device="cuda", generator=g).to(torch.bfloat16)
    xs = [torch.randn(max(1, c // 1024), tokens, device="cuda", generator=g).to(torch.bfloat16) for _, c in plan]
    outs = [torch.empty(x.shape[0], 1024, device="cuda", dtype=torch.bfloat16) for x in xs]
    cs, ms_normal = torch.cuda.Stream(), torch.cuda.Stream()
    # a high-priority communication stream: its CTAs are scheduled ahead of queued GEMM CTAs
    lo, hi = torch.cuda.Stream.priority_range() if hasattr(torch.cuda.Stream, "priority_range") else (0, -1)
    ms_high = torch.cuda.Stream(priority=hi)
    main = torch.cuda.current_stream()

    def compute(events=None):
        for b, x in enumerate(xs):
            torch.matmul(x, gy, out=outs[b])
            if events is not None:
                events[b].record(torch.cuda.current_stream())

    def timed(fn, reps=5):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(main)
        for _ in range(reps):
            fn()
        b.record(main)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    def compute_only():
        cs.wait_stream(main)
        with torch.cuda.stream(cs):
            compute()
        main.wait_stream(cs)

    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def comm_only(max_sms, engine, ms):
        ms.wait_stream(main)
        ra.ra_allreduce_buckets(sends, recvs, plan, op, max_sms=max_sms, engine=engine, status=status, stream=ms)
        main.wait_stream(ms)

    def overlapped(max_sms, engine, ms):
        events = [torch.cuda.Event() for _ in plan]
        cs.wait_stream(main)
        ms.wait_stream(main)
        with torch.cuda.stream(cs):
            compute(events)
        ra.ra_allreduce_buckets(sends, recvs, plan, op, ready_events=events, max_sms=max_sms, engine=engine,
                                status=status, stream=ms)
        main.wait_stream(cs)
        main.wait_stream(ms)

    def overlapped_on(cs_, ms_, engine="registers"):
        events = [torch.cuda.Event() for _ in plan]
        cs_.wait_stream(main)
        ms_.wait_stream(main)
        with torch.cuda.stream(cs_):
            compute(events)
        ra.ra_allreduce_buckets(sends, recvs, plan, op, ready_events=events, engine=engine, status=status,
                                stream=ms_)
        main.wait_stream(cs_)
        main.wait_stream(ms_)

    c_ms = timed(compute_only)
    flops = sum(2 * c * tokens for _, c in plan)
    s_bytes = length * 2
    runs = [(e, m, "normal") for e in ("registers", "bulk") for m in (0, 76, 38, 16, 8)]
    runs += [(e, m, "high") for e in ("registers", "bulk") for m in (0, 76)]
    for engine, max_sms, prio in runs:
        ms = ms_high if prio == "high" else ms_normal
        a_ms = timed(lambda: comm_only(max_sms, engine, ms))
        t_ms = timed(lambda: overlapped(max_sms, engine, ms))
        rec = {"mode": "overlap", "workload": "ar_n8_bf16_avg_gpt2m", "buckets": len(plan),
               "bucket_cap_bytes": 25 * 1000 * 1000, "tokens": tokens, "engine": engine, "max_sms": max_sms,
               "comm_stream_priority": prio,
               "compute_ms": round(c_ms, 3), "compute_tflops": round(flops / (c_ms * 1e-3) / 1e12, 1),
               "allreduce_ms": round(a_ms, 3), "allreduce_algbw_GBps": round(s_bytes / (a_ms * 1e-3) / GB, 1),
               "overlapped_ms": round(t_ms, 3), "exposed_comm_ms": round(t_ms - c_ms, 3),
               "hidden_fraction": round((c_ms + a_ms - t_ms) / a_ms, 3), "status": int(status.item())}
        print(json.dumps(rec), flush=True)

    # SM partitions: the GEMMs on one green context, the all-reduces on another with k SMs
    a_all = timed(lambda: comm_only(0, "registers", ms_normal))
    for k in (16, 32, 48, 64, 96):
        try:
            (ms_k, k_sms), (cs_k, rest_sms) = green_partition(k)
        except RuntimeError as e:  # no green contexts here: say so and stop the sweep
            print(json.dumps({"mode": "overlap_split", "unavailable": str(e)}), flush=True)
            break
        for engine in ("registers", "bulk"):
            def comm_k():
                ms_k.wait_stream(main)
                ra.ra_allreduce_buckets(sends, recvs, plan, op, engine=engine, status=status, stream=ms_k)
                main.wait_stream(ms_k)

            def compute_k():
                cs_k.wait_stream(main)
                with torch.cuda.stream(cs_k):
                    compute()
                main.wait_stream(cs_k)

            a_k = timed(comm_k)
            c_k = timed(compute_k)
            t_k = timed(lambda: overlapped_on(cs_k, ms_k, engine))
            rec = {"mode": "overlap_split", "workload": "ar_n8_bf16_avg_gpt2m", "buckets": len(plan), "tokens": tokens,
                   "engine": engine, "comm_sms": k_sms, "compute_sms": rest_sms,
                   "allreduce_ms_on_comm_sms": round(a_k, 3),
                   "allreduce_hbm_GBps_per_comm_sm": round(2 * n * s_bytes / (a_k * 1e-3) / GB / k_sms, 1),
                   "compute_ms_on_compute_sms": round(c_k, 3), "overlapped_ms": round(t_k, 3),
                   "unsplit_compute_ms": round(c_ms, 3), "unsplit_allreduce_ms": round(a_all, 3),
                   "hidden_fraction": round((c_ms + a_all - t_k) / a_all, 3), "status": int(status.item())}
            print(json.dumps(rec), flush=True)
    return 0


_green = {}


def green_partition(k):
    """Two CUDA green contexts on device 0: one with k SMs, one with the rest; a stream on each.
    Returns ((stream_k, sms_k), (stream_rest, sms_rest)). Driver API through ctypes."""
    import ctypes

    import torch

    if k in _green:
        return _green[k]
    cu = ctypes.CDLL("libcuda.so.1")

    def ck(res, what):
        if res != 0:
            raise RuntimeError(f"{what} failed (CUresult {res})")

    dev = ctypes.c_int()
    ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
    Res = ctypes.c_ubyte * 144  # CUdevResource: type, 92 bytes of padding, then the SM counts
    whole, part, rest = Res(), Res(), Res()
    ck(cu.cuDeviceGetDevResource(dev, ctypes.byref(whole), 1), "cuDeviceGetDevResource")
    nb = ctypes.c_uint(1)
    ck(cu.cuDevSmResourceSplitByCount(ctypes.byref(part), ctypes.byref(nb), ctypes.byref(whole), ctypes.byref(rest),
                                      0, k), "cuDevSmResourceSplitByCount")
    out = []
    for r in (part, rest):
        desc, ctx, stream = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
        ck(cu.cuDevResourceGenerateDesc(ctypes.byref(desc), ctypes.byref(r), 1), "cuDevResourceGenerateDesc")
        ck(cu.cuGreenCtxCreate(ctypes.byref(ctx), desc, dev, 1), "cuGreenCtxCreate")
        ck(cu.cuGreenCtxStreamCreate(ctypes.byref(stream), ctx, 1, 0), "cuGreenCtxStreamCreate")
        out.append((torch.cuda.ExternalStream(stream.value), int.from_bytes(bytes(r[96:100]), "little")))
    _green[k] = tuple(out)
    return _green[k]


# ---------------------------------------------------------------------------
# stream roofs (not the headline): what HBM gives to reads and to writes from
# persistent and from one-shot CTAs, beside torch's copy and fill and the
# library's all-gather
# ---------------------------------------------------------------------------
def run_roofs(args):
    import ctypes

    import torch

    from ring_all_reduce_02_gb300 import build, ra

    build.build()
    probe = ctypes.CDLL(build.build_probe())
    probe.rp_store.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.c_size_t,
                               ctypes.c_void_p]
    probe.rp_load.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]
    probe.rp_copy.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    probe.rp_copy_sms.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
    probe.rp_copy_n.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.c_size_t,
                                ctypes.c_void_p]
    probe.rp_read_n.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                ctypes.c_void_p]
    torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    peak, peak_kind = measured_peaks()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(int(2 * l2), dtype=torch.uint8, device="cuda")
    evict = torch.ones(int(2 * l2) // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    total = 4 << 30
    big = torch.empty(total, dtype=torch.uint8, device="cuda")
    other = torch.empty(total // 2, dtype=torch.uint8, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")

    def check(rc):
        if rc:
            raise RuntimeError(f"stream probe failed: cudaError {rc}")

    def store(one_shot, bufs):
        arr = (ctypes.c_void_p * len(bufs))(*[b.data_ptr() for b in bufs])
        return lambda: check(probe.rp_store(one_shot, arr, len(bufs), bufs[0].numel(), stream.cuda_stream))

    def load(one_shot, buf):
        return lambda: check(probe.rp_load(one_shot, buf.data_ptr(), buf.numel(), sink.data_ptr(), stream.cuda_stream))

    def timed(fn, nbytes, label, extra=None, sms=0):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        clean = []
        for _ in range(10):  # each launch from an L2 of clean, unrelated lines
            flush.zero_()
            torch.amax(evict)
            torch.cuda._sleep(200_000)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            clean.append(a.elapsed_time(b) * 1e-3)
        torch.cuda._sleep(200_000)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 10
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        b2b = a.elapsed_time(b) * 1e-3 / reps
        rec = {"mode": "roofs", "what": label, "bytes": nbytes,
               "clean_GBps": round(nbytes / statistics.median(clean) / GB, 1),
               "b2b_GBps": round(nbytes / b2b / GB, 1),
               "b2b_frac_of_copy_peak": round(nbytes / b2b / GB / peak, 4), "peak": f"{peak} ({peak_kind})"}
        if sms:
            rec["sms"] = sms
            rec["b2b_GBps_per_sm"] = round(nbytes / b2b / GB / sms, 1)
        rec.update(extra or {})
        print(json.dumps(rec), flush=True)

    sampler = ClockSampler(dev).start()
    time.sleep(0.3)
    t0 = time.time()
    f32 = big.view(torch.float32)
    timed(lambda: other.view(torch.float32).copy_(f32[: total // 8]), total, "torch copy_ (read 2 GiB + write 2 GiB)")
    timed(lambda: f32.fill_(1.5), total, "torch fill_ (write 4 GiB)")
    timed(store(0, [big]), total, "store stream, persistent CTAs (write 4 GiB)")
    timed(store(1, [big]), total, "store stream, one-shot CTAs (write 4 GiB)")
    timed(load(0, big), total, "load stream, persistent CTAs (read 4 GiB)")
    timed(load(1, big), total, "load stream, one-shot CTAs (read 4 GiB)")
    for one_shot, style in ((0, "persistent"), (1, "one-shot")):
        timed(lambda: check(probe.rp_copy(one_shot, big.data_ptr(), other.data_ptr(), total // 2, stream.cuda_stream)),
              total, f"copy, {style} CTAs (read 2 GiB + write 2 GiB)")
    n8, l8 = 8, (256 << 20) // 4
    s8 = [torch.randn(l8, device="cuda") for _ in range(n8)]
    r8 = [torch.empty_like(x) for x in s8]
    timed(lambda: ra.ra_allreduce(s8, r8, "avg", stream=stream), 2 * n8 * l8 * 4,
          "library all-reduce, N = 8, fp32 avg, 256 MiB per rank (the bench workload)", {"nranks": n8})
    # what a share of the SMs can move: a plain copy on k CTAs of 1024 threads (one per SM), and the
    # library's all-reduce on an SM budget of k with either engine
    bstat = torch.zeros(1, dtype=torch.int32, device="cuda")
    for k in (16, 32, 64):
        nb = k * (16 << 20)
        timed(lambda: check(probe.rp_copy_sms(big.data_ptr(), other.data_ptr(), nb // 2, k, stream.cuda_stream)),
              nb, f"copy on {k} SMs (one 1024-thread CTA per SM)", sms=k)
        for engine in ("registers", "bulk"):
            timed(lambda: ra.ra_allreduce_ex(s8, r8, "avg", max_sms=k, engine=engine,
                                             status=bstat if engine == "bulk" else None, stream=stream),
                  2 * n8 * l8 * 4, f"library all-reduce on {k} SMs, {engine} engine, N = 8, fp32 avg, 256 MiB per rank",
                  {"nranks": n8}, sms=k)
    if bstat.item() != 0:
        raise RuntimeError(f"bulk engine reported status {bstat.item()}")
    del s8, r8
    for n in (8, 16):
        bufs = [big[r * (total // n):(r + 1) * (total // n)] for r in range(n)]
        timed(store(0, bufs), total, f"store stream to {n} buffers, persistent CTAs (write 4 GiB)")
        timed(store(1, bufs), total, f"store stream to {n} buffers, one-shot CTAs (write 4 GiB)")
        # the all-gather's mix: each piece read once from `other` and written to the n buffers
        piece = total // n
        arr = (ctypes.c_void_p * n)(*[b.data_ptr() for b in bufs])
        timed(lambda: check(probe.rp_copy_n(other.data_ptr(), arr, n, piece, stream.cuda_stream)), piece + total,
              f"read once, write to {n} buffers, one-shot CTAs (read {piece >> 20} MiB + write 4 GiB)")
        # the reduce-scatter's mix: each piece read from the n buffers, one combination written to `other`
        timed(lambda: check(probe.rp_read_n(arr, n, other.data_ptr(), piece, stream.cuda_stream)), total + piece,
              f"read {n} buffers, write once, one-shot CTAs (read 4 GiB + write {piece >> 20} MiB)")
        rs_len = (1 << 30) // 4 // n
        rs_in = [torch.randn(rs_len, device="cuda") for _ in range(n)]
        rs_bounds = [ra.ra_chunk_range(rs_len, n, c) for c in range(n)]
        rs_out = [torch.empty(e - b, device="cuda") for b, e in rs_bounds]
        timed(lambda: ra.ra_reduce_scatter(rs_in, rs_out, "sum", stream=stream), (n + 1) * rs_len * 4,
              f"library reduce-scatter, N = {n}, fp32 sum, 1 GiB over all ranks", {"nranks": n})
        del rs_in, rs_out
        length = (1 << 30) // 4 // n
        bounds = [ra.ra_chunk_range(length, n, c) for c in range(n)]
        shards = [torch.randn(e - b, device="cuda") for b, e in bounds]
        recvs = [torch.empty(length, device="cuda") for _ in range(n)]
        timed(lambda: ra.ra_allgather(shards, recvs, stream=stream), (n + 1) * length * 4,
              f"library all-gather, N = {n}, fp32, 1 GiB over all ranks", {"nranks": n})
        del shards, recvs
    t1 = time.time()
    time.sleep(0.2)
    sampler.stop()
    print(json.dumps({"mode": "roofs", "clocks": sampler.summary(t0, t1)}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", default=None, help="write the message-size sweep to this JSONL file")
    ap.add_argument("--sweep-max", type=int, default=0, help="largest count in the sweep (0 = all)")
    ap.add_argument("--overlap", action="store_true", help="bucketed all-reduce beside a synthetic backward")
    ap.add_argument("--overlap-tokens", type=int, default=2048)
    ap.add_argument("--call", default=None, choices=sorted(CALLS),
                    help="time one call alone on the workload (per-kernel roofline; not the headline)")
    ap.add_argument("--roofs", action="store_true",
                    help="stream roofs: reads and writes from persistent and one-shot CTAs (not the headline)")
    ap.add_argument("--case", default=None, metavar="N,COUNT,DTYPE,OP",
                    help="with --call: this case instead of the named workload (e.g. 16,16777216,f32,sum)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.overlap:
        return run_overlap(args)
    if args.roofs:
        return run_roofs(args)
    if args.call:
        return run_call(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
