"""Benchmark of the ZeRO-1 step for N simulated ranks on one GB300.

    python bench.py [--gpus G] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...       # the CPU oracle as the reference arm

Prints one JSON line.  `value` is whole-job throughput in GB/s of algorithmic
bytes (N*P gradient reads + 24*P master/m/v read and write + N*P weight writes
per step, the minimum the step must move), with every input resident in HBM.
`e2e` is the same metric end to end through the public API with the step's
gradients copied from pinned host memory and the global norm read back, every
step.  `roofline` covers the dominant kernel, timed with CUDA events on its own
launch stream inside the timed region.  `cpu_baseline` is the CPU oracle on a
bounded window of the same workload.

With G > 1 (torchrun, one process per GPU) every rank runs its own replica of
the workload: the step has no cross-GPU exchange, so scaling is weak and
`value` sums all ranks' bytes over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import inputs as I  # noqa: E402

METRIC = "ZeRO-1 step GB/s and % of GB300 HBM roofline; steps/s vs CPU oracle"
UNIT = "GB/s"
DEFAULT_WORKLOAD = I.GPT2_1P5B.name
PROFILES = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "gradient_reduction_zero_gb300", "csrc")
# The translation unit of each kernel whose DRAM traffic profiles/ncu_traffic.json
# holds: its .cu file and the headers it includes.  The traffic of a kernel is
# used only while these sources (and the nvcc flags) hash as they did when the
# counters were taken.
KERNEL_UNITS = {
    "dpz_rs_avg_sumsq": ("device.cuh", "internal.h", "reduce.cu"),
    "dpz_adamw_bcast": ("bulk.cuh", "device.cuh", "internal.h", "staged.cu"),
    "dpz_zero1_fused_sumsq": ("bulk.cuh", "device.cuh", "internal.h", "staged.cu"),
    "dpz_norm_owned": ("bulk.cuh", "device.cuh", "internal.h", "staged.cu"),
}


# ------------------------------------------------------------------ bytes

def step_bytes(w: I.Workload) -> int:
    """Algorithmic bytes of one step (the minimum it must move)."""
    eg, ew = w.grad_bytes(), w.weight_bytes()
    if w.allreduce_only:
        return 2 * w.N * w.P * eg
    return w.N * w.P * eg + 24 * w.P + w.N * w.P * ew


def kernel_bytes(name: str, w: I.Workload) -> int:
    """Algorithmic bytes of one launch of each kernel."""
    N, P, eg, ew = w.N, w.P, w.grad_bytes(), w.weight_bytes()
    return {
        "dpz_rs_avg_sumsq": N * P * eg + P * eg,
        "dpz_rs_avg": N * P * eg + P * eg,
        "dpz_adamw_bcast": P * eg + 24 * P + N * P * ew,
        "dpz_adamw_owner": P * eg + 24 * P + P * ew,
        "dpz_zero1_fused": N * P * eg + 24 * P + N * P * ew,
        "dpz_zero1_fused_sumsq": N * P * eg + 24 * P + N * P * ew,
        "dpz_allreduce_avg": 2 * N * P * eg,
        "dpz_allgather": N * P * ew,
        "dpz_norm_owned": P * eg,
        "dpz_norm_finalize": 8 * N * ((P // N + 255) // 256),
    }.get(name, 0)


def peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def kernel_source_hash(kernel: str) -> str:
    """Hash of one kernel's translation unit (KERNEL_UNITS) with comments and
    whitespace removed, and of the nvcc flags: it changes when the code does,
    not when only a comment does."""
    from gradient_reduction_zero_gb300 import build as B
    h = hashlib.sha256()
    for p in (os.path.join(CSRC, f) for f in KERNEL_UNITS[kernel]):
        with open(p, encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    h.update(" ".join(f for f in B.NVCC_FLAGS if not f.startswith("-I")).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, w: I.Workload):
    """DRAM bytes per launch from the committed ncu summary, scaled to this
    workload by the units processed; None if absent or the kernels changed."""
    path = os.path.join(PROFILES, "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    k = t.get("kernels", {}).get(kernel)
    if not k or kernel not in KERNEL_UNITS or k.get("source_hash") != kernel_source_hash(kernel):
        return None
    if (k.get("N"), k.get("gdtype"), k.get("wdtype")) != (w.N, w.gdtype, w.wdtype):
        return None
    return int(k["dram_bytes_per_element"] * w.P)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
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
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t_lo: float, t_hi: float) -> dict | None:
        """Summary of the samples taken between host times t_lo and t_hi."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in self.lines:
            if ts < t_lo or ts > t_hi:
                continue
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


REJECTING_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_rejected(clk: dict | None) -> bool:
    """True for a timed region whose clock record makes it invalid: a
    hardware or thermal slowdown was active, or the SM clock sat well below
    its maximum with no reason given (a clock locked by someone else).  The
    power cap alone is kept (normal on a 1.4 kW part) and only noted."""
    if not clk:
        return False
    if any(r in clk.get("reasons", ()) for r in REJECTING_REASONS):
        return True
    return not clk.get("reasons") and clk["sm_mhz"] < 0.85 * clk["sm_max_mhz"]


# ------------------------------------------------------------------ ranks

def dist_setup(gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)      # each rank's collectives on its own GPU
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle

def oracle_window_step(w: I.Workload, width: int, offset: int = 0):
    """Inputs for one oracle step on a window of `width` elements of every
    chunk (a mini-arena of N*width elements per rank), generated up front."""
    g = I.window_arena_host(w, offset, width)
    th = I.window_state_host(w, "master", offset, width)
    m = I.window_state_host(w, "m", offset, width)
    v = I.window_state_host(w, "v", offset, width)
    wt = np.zeros((w.N, w.N * width), dtype=np.uint16 if w.wdtype == "bf16" else np.float32)
    return g, th, m, v, wt


def time_oracle(w: I.Workload, seconds: float) -> dict:
    """The oracle as it stands, single-threaded, on windows of the workload
    until about `seconds` of CPU time; throughput in the metric's unit."""
    import oracle as O
    width = min(w.C, 1 << 18)
    cfg = O.cfg_from_workload(w)
    mini = w.with_(P=w.N * width)
    base = oracle_window_step(w, width, offset=(w.C - width) // 2)
    done_bytes, elapsed, reps = 0, 0.0, 0
    while elapsed < seconds or reps == 0:
        args = [a.copy() for a in base]
        t0 = time.perf_counter()
        if w.allreduce_only:
            O.ring_allreduce_avg(args[0])
        else:
            # the window's own norm stands in for the arena's: same work
            O.zero1_step(*args, cfg)
        elapsed += time.perf_counter() - t0
        done_bytes += step_bytes(mini)
        reps += 1
    return {"value": done_bytes / elapsed / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "steps_per_s": done_bytes / elapsed / step_bytes(w),
            "sample": f"{reps} windows of {width} elements per chunk x {w.N} chunks x {w.N} ranks "
                      f"of {w.name} ({elapsed:.1f} s single-threaded)"}


def oracle_thread_windows(w: I.Workload, threads: int) -> list:
    """Inputs of `threads` disjoint windows of the workload, one per thread."""
    width = min(w.C, 1 << 18)
    span = max(1, (w.C - width) // max(1, threads))
    return [oracle_window_step(w, width, offset=min(w.C - width, t * span) // 8 * 8)
            for t in range(threads)]


def time_oracle_threads(w: I.Workload, seconds: float, threads: int, bases=None) -> dict:
    """The same oracle, unchanged, on `threads` disjoint windows of the
    workload at once, one host thread each (the oracle's C calls release the
    GIL), for about `seconds` of wall time; throughput in the metric's unit.
    `bases`: the windows' inputs from oracle_thread_windows, to reuse."""
    import threading
    import oracle as O
    width = min(w.C, 1 << 18)
    cfg = O.cfg_from_workload(w)
    mini = w.with_(P=w.N * width)
    if bases is None:
        bases = oracle_thread_windows(w, threads)
    counts = [0] * threads
    start = threading.Barrier(threads + 1)
    stop = threading.Event()

    def work(t):
        start.wait()
        while not stop.is_set() or counts[t] == 0:
            args = [a.copy() for a in bases[t]]
            if w.allreduce_only:
                O.ring_allreduce_avg(args[0])
            else:
                O.zero1_step(*args, cfg)
            counts[t] += 1

    pool = [threading.Thread(target=work, args=(t,)) for t in range(threads)]
    for th in pool:
        th.start()
    start.wait()
    t0 = time.perf_counter()
    time.sleep(seconds)
    stop.set()
    for th in pool:
        th.join()
    elapsed = time.perf_counter() - t0
    done = sum(counts)
    return {"value": done * step_bytes(mini) / elapsed / 1e9, "unit": UNIT, "cores": threads,
            "kind": "oracle", "steps_per_s": done * step_bytes(mini) / elapsed / step_bytes(w),
            "sample": f"{done} windows of {width} elements per chunk x {w.N} chunks x {w.N} ranks "
                      f"of {w.name} on {threads} host threads, disjoint windows "
                      f"({elapsed:.1f} s wall)"}


def run_reference(args) -> None:
    """The CPU oracle timed as the reference arm: rank 0 only, the unchanged
    oracle on disjoint windows of the workload, one per host core, each step a
    bounded slice of wall time, the whole run kept to a few minutes."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    w = I.WORKLOADS[args.workload]
    threads = os.cpu_count() or 1
    bases = oracle_thread_windows(w, threads)
    per_step = []
    secs = min(args.ref_seconds, 150.0 / max(1, args.warmup + args.steps))
    for i in range(args.warmup + args.steps):
        r = time_oracle_threads(w, secs, threads, bases)
        if i >= args.warmup:
            per_step.append(r)
    vals = [r["value"] for r in per_step]
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_bytes(w) / (value * 1e9) * 1e3,
            "steps_per_s": value * 1e9 / step_bytes(w),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": per_step[-1]["sample"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


L2_BYTES = 129e6
# groups of consecutive steps whose median time per step is reported
TIMING_REPS = 20


def touched_bytes(w: I.Workload) -> int:
    """Device bytes one step reads or writes: the gradient arena for an
    all-reduce; gradients, weights and master/m/v for the step."""
    if w.allreduce_only:
        return w.N * w.P * w.grad_bytes()
    return w.N * w.P * (w.grad_bytes() + w.weight_bytes()) + 12 * w.P


def l2_note(w: I.Workload) -> str:
    b = touched_bytes(w)
    if b > 2 * L2_BYTES:
        return "inputs larger than L2 (%.2f GB touched per step vs 129 MB L2)" % (b / 1e9)
    return ("arena within reach of L2 (%.1f MB touched per step vs 129 MB L2): no flush "
            "between steps, so the figures include L2 reuse" % (b / 1e6))


def config_of(w: I.Workload, acc32: bool = False) -> dict:
    c = {"workload": w.name, "ranks_simulated": w.N, "P": w.P,
         "grad_dtype": w.gdtype + ("+fp32-accumulate" if acc32 else ""),
         "weight_dtype": w.wdtype, "state_dtype": "f32" if not w.allreduce_only else None,
         "clip": w.clip, "step_t": w.step,
         "l2": l2_note(w),
         "parallelism": f"{w.N} simulated ranks per GPU"}
    return c


# ------------------------------------------------------------------ GPU arm

def allocate(w: I.Workload, dev):
    import torch
    gd = torch.bfloat16 if w.gdtype == "bf16" else torch.float32
    wd = torch.bfloat16 if w.wdtype == "bf16" else torch.float32
    G = torch.empty(w.N * w.P, dtype=gd, device=dev)
    I.fill_grads_device(w, G)
    if w.allreduce_only:
        return G, None, None, None, None
    T = torch.empty(w.P, dtype=torch.float32, device=dev)
    M = torch.empty_like(T)
    V = torch.empty_like(T)
    for which, t in (("master", T), ("m", M), ("v", V)):
        I.fill_state_device(w, which, t)
    W = torch.zeros(w.N * w.P, dtype=wd, device=dev)
    return G, T, M, V, W


ENTRIES = ("step", "reduce_scatter", "allreduce", "norm", "adamw_owner", "allgather", "update",
           "range", "bucket_zero2", "norm_static")


def entry_bytes(entry: str, w: I.Workload) -> int:
    """Algorithmic bytes of one call of a single entry point."""
    N, P, eg, ew = w.N, w.P, w.grad_bytes(), w.weight_bytes()
    return {"reduce_scatter": N * P * eg + P * eg,
            "range": N * P * eg + P * eg,
            "bucket_zero2": N * P * eg + P * eg,
            "allreduce": 2 * N * P * eg,
            "norm": P * eg, "norm_static": P * eg,
            "adamw_owner": P * eg + 24 * P + P * ew,
            "update": P * eg + 24 * P + N * P * ew,
            "allgather": N * P * ew}[entry]


def entry_op(args, w, dpz, G, T, M, V, W, ws, nrm, cfg, stream):
    """One entry point alone, on the workload's buffers (for per-kernel timing
    and profiling).  Every call computes real results from the previous one's
    buffers; the bytes are the same each time."""
    import torch
    N, P = w.N, w.P
    if args.entry == "bucket_zero2":
        shards = torch.empty(P, dtype=G.dtype, device=G.device)
    if args.entry == "allreduce":
        return lambda on=None: dpz.dp_allreduce_avg(G, N, on or stream, acc32=args.acc32)
    if args.entry == "reduce_scatter":
        return lambda on=None: dpz.dp_reduce_scatter_avg(G, N, on or stream, acc32=args.acc32)
    if args.entry == "range":
        return lambda on=None: dpz.dp_reduce_scatter_avg_range(G, N, 0, P, ws=ws,
                                                               stream=on or stream,
                                                               acc32=args.acc32)
    if args.entry == "bucket_zero2":
        # the whole arena as one bucket: staging = the arena, shards = [P]
        return lambda on=None: dpz.dp_reduce_scatter_avg_bucket(G, 0, shards, N, ws=ws,
                                                                stream=on or stream,
                                                                acc32=args.acc32)
    if args.entry == "norm":
        return lambda on=None: dpz.dp_grad_global_norm(G, N, ws, nrm, stream=on or stream)
    if args.entry == "norm_static":
        return lambda on=None: dpz.dp_grad_global_norm_static(G, N, nrm, stream=on or stream)
    if args.entry == "adamw_owner":
        return lambda on=None: dpz.zero1_adamw_step(G, T, M, V, W, N, cfg, ws=ws,
                                                    stream=on or stream)
    if args.entry == "update":
        return lambda on=None: dpz.dp_zero1_update(G, T, M, V, W, N, cfg, ws=ws,
                                                   stream=on or stream)
    if args.entry == "allgather":
        return lambda on=None: dpz.dp_allgather(W, N, on or stream)
    raise ValueError(args.entry)


def run_gpu(args) -> None:
    import torch

    world, rank, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import gradient_reduction_zero_gb300.dpz as dpz

    w = I.WORKLOADS[args.workload]
    if args.clip is not None:
        w = w.with_(clip=args.clip)
    G, T, M, V, W = allocate(w, dev)
    ws = dpz.workspace(w.P, w.N, dev)
    nrm = torch.zeros(1, dtype=torch.float32, device=dev)
    cfg = dpz.make_cfg(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.step, w.clip)
    stream = torch.cuda.current_stream()

    def step_with(grads, on):
        if w.allreduce_only:
            dpz.dp_allreduce_avg(grads, w.N, on, acc32=args.acc32)
        else:
            dpz.dp_zero1_step(grads, T, M, V, W, w.N, cfg, ws=ws, norm_out=nrm, stream=on,
                              acc32=args.acc32)

    def full_step(on=None):
        step_with(G, stream if on is None else on)

    step = full_step
    if args.entry != "step":
        # one full step first leaves a valid norm in the workspace
        if not w.allreduce_only:
            full_step()
        step = entry_op(args, w, dpz, G, T, M, V, W, ws, nrm, cfg, stream)
        args.no_e2e = args.no_cpu_baseline = True
        args.buckets = 0

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    # ---------------------------------------------------------------- timed
    # The K steps in REPS groups of consecutive steps (one step per group when
    # K <= REPS), a CUDA event on the launch stream before the first group and
    # after every group: ms_per_step is the median over the groups of the
    # group's time per step, the mean is reported beside it.  Groups keep the
    # events' own host cost out of launch-bound steps of a few microseconds.
    # The library's per-kernel event pairs stay off here; they come from the
    # separate pass below.
    reps = min(args.steps, TIMING_REPS)
    sizes = [args.steps // reps + (1 if g < args.steps % reps else 0) for g in range(reps)]

    def timed_region():
        clocks = ClockSampler(local)
        clocks.start()
        time.sleep(0.5)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        launches0 = dpz.launch_count()
        barrier(world)
        torch.cuda.synchronize()
        t_lo = time.time()
        ev[0].record(stream)
        for g, n in enumerate(sizes):
            for _ in range(n):
                step()
            ev[g + 1].record(stream)
        torch.cuda.synchronize()
        t_hi = time.time()
        barrier(world)
        launches = dpz.launch_count() - launches0
        time.sleep(0.2)
        clk = clocks.stop(t_lo, t_hi)
        per_step = [ev[g].elapsed_time(ev[g + 1]) / n for g, n in enumerate(sizes)]
        return per_step, ev[0].elapsed_time(ev[-1]) / args.steps, launches, clk

    per_step, mean_ms, launches, clk = timed_region()
    remeasured = None
    if max_over_ranks(1.0 if clocks_rejected(clk) else 0.0, world) > 0.0:
        # a throttled or clock-locked timed region is taken again, once
        remeasured = {"first_ms_per_step": round(statistics.median(per_step), 5),
                      "first_clocks": clk}
        per_step, mean_ms, launches, clk = timed_region()
    ms = statistics.median(per_step)
    ms_max = max_over_ranks(ms, world)
    ms_mean = max_over_ranks(mean_ms, world)
    spread = [round(min(per_step), 5), round(max(per_step), 5)]

    nbytes = step_bytes(w) if args.entry == "step" else entry_bytes(args.entry, w)
    value = nbytes * world / (ms_max * 1e-3) / 1e9
    pk = peaks()

    # ------------------------------------------------- per-kernel times
    # The same steps again with the library's event pair around each of its
    # launches: each kernel's average duration and its share of the step.
    barrier(world)
    torch.cuda.synchronize()
    dpz.profile_start(16 * args.steps + 16)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    kstats = dpz.profile_stop()

    # dominant kernel: largest share of the profiled pass
    dom = max(kstats.items(), key=lambda kv: kv[1][1])
    dname, (dn, dms) = dom
    per_launch_ms = dms / dn
    kb = kernel_bytes(dname, w) if args.entry == "step" else entry_bytes(args.entry, w)
    achieved = kb / (per_launch_ms * 1e-3) / 1e9
    shares = {k: {"launches": n, "ms_total": round(t, 4),
                  "share": round(t / sum(x[1] for x in kstats.values()), 4)}
              for k, (n, t) in kstats.items()}

    # ---------------------------------------------------------------- buckets
    bucketed = None
    if args.buckets and not w.allreduce_only:
        rs = kstats.get("dpz_rs_avg_sumsq") or kstats.get("dpz_zero1_fused_sumsq")
        bucketed = run_buckets(args, w, G, T, M, V, W, ws, nrm, cfg, stream, rs[1] / rs[0])

    # ---------------------------------------------------------------- graph
    graph = None
    if args.graph:
        graph = run_graph(args, step, stream, world, nbytes)

    # ------------------------------------------- prepared call (host cost)
    # Launch-bound steps: the same K steps through a PreparedCall (arguments
    # marshalled once, the library still validating and launching every time)
    # show how much of a step's time is the Python wrapper's.
    prepared = None
    if args.entry == "step" and touched_bytes(w) < L2_BYTES:
        if w.allreduce_only:
            call = dpz.prepare_allreduce_avg(G, w.N, stream, acc32=args.acc32)
        else:
            call = dpz.prepare_zero1_step(G, T, M, V, W, w.N, cfg, ws=ws, norm_out=nrm,
                                          stream=stream, acc32=args.acc32)
        for _ in range(max(3, args.warmup)):
            call()
        torch.cuda.synchronize()
        pe = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        pe[0].record(stream)
        for g, n in enumerate(sizes):
            for _ in range(n):
                call()
            pe[g + 1].record(stream)
        torch.cuda.synchronize()
        pms = statistics.median(pe[g].elapsed_time(pe[g + 1]) / n for g, n in enumerate(sizes))
        prepared = {"ms_per_step": round(pms, 5), "steps_per_s": round(1e3 / pms, 1),
                    "how": "the same steps through dpz.prepare_zero1_step / "
                           "prepare_allreduce_avg: arguments marshalled once, the C-ABI "
                           "call (validation and launch) made every step"}

    # ---------------------------------------------------------------- e2e
    e2e = None
    if not args.no_e2e:
        full = None if w.allreduce_only or w.clip <= 0 else (T, M, V, W, ws, cfg)
        e2e = run_e2e(args, w, G, step_with, nrm, stream, world, full)

    # ------------------------------------------------ the other workloads
    configs = None
    if world == 1 and not args.no_configs and args.entry == "step" \
            and args.workload == DEFAULT_WORKLOAD and args.clip is None:
        del G, T, M, V, W
        torch.cuda.empty_cache()
        configs = measure_configs(args, dev, stream)

    cpu = cpu_mt = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = time_oracle(w, args.cpu_seconds)
        cpu_mt = time_oracle_threads(w, args.cpu_seconds, os.cpu_count() or 1)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(ms_max, 4),
            "ms_per_step_mean": round(ms_mean, 4),
            "ms_per_step_min_max": spread,
            "timing": f"median over {reps} groups of {sizes[0]} consecutive steps of the time "
                      "per step between CUDA events on the launch stream; kernel times from a "
                      "separate profiled pass of the same steps",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": dict(config_of(w, args.acc32), entry=args.entry),
            "steps_per_s": round(1e3 / ms_max, 3),
            "pct_of_hbm_roofline": {
                "measured_copy_peak": round(100 * value / world / pk["hbm_gbs"], 2),
                "spec_8tbs": round(100 * value / world / 8000.0, 2)},
            "bytes_per_step": nbytes,
            "roofline": {"bound": "hbm", "kernel": dname, "achieved": round(achieved, 1),
                         "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / pk["hbm_gbs"], 4),
                         "traffic": ncu_traffic(dname, w),
                         "algorithmic_bytes_per_launch": kb,
                         "ms_per_launch": round(per_launch_ms, 4),
                         "peak_source": pk["source"] + " (MEASURED_PEAKS.json hbm_gbs)"},
            "kernels": shares,
            "gpu_launches": launches,
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "cpu_baseline_threads": cpu_mt,
        }
        if remeasured is not None:
            line["remeasured"] = remeasured
        if graph is not None:
            line["graph_replay"] = graph
        if prepared is not None:
            line["prepared_call"] = prepared
        if configs is not None:
            line["configs"] = configs
        if bucketed is not None:
            line["bucket_overlap"] = bucketed
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def time_median(fn, stream, steps: int) -> float:
    """fn() `steps` times in min(steps, TIMING_REPS) groups of consecutive
    calls, a CUDA event on `stream` before the first group and after each:
    the median over the groups of the time per call, in ms."""
    import torch
    reps = min(steps, TIMING_REPS)
    sizes = [steps // reps + (1 if g < steps % reps else 0) for g in range(reps)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    for g, n in enumerate(sizes):
        for _ in range(n):
            fn()
        ev[g + 1].record(stream)
    torch.cuda.synchronize()
    return statistics.median(ev[g].elapsed_time(ev[g + 1]) / n for g, n in enumerate(sizes))


def warm_up(fn, stream, calls: int, min_ms: float = 20.0) -> None:
    """`calls` calls of fn, then more until about min_ms of device time has
    passed in all: right after a large buffer is freed, a new one can run
    below speed for a few milliseconds (measured: an all-reduce of 2 x 256 MiB
    took 188 us per call over its first 20 calls after a 56 GB buffer was
    freed, against 157 us fresh)."""
    import torch
    for _ in range(calls):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    fn()
    e1.record(stream)
    torch.cuda.synchronize()
    one = max(e0.elapsed_time(e1), 1e-3)
    for _ in range(min(int(min_ms / one), 10000)):
        fn()


def measure_configs(args, dev, stream) -> dict:
    """The other workloads, timed on the device as the headline is (median
    over groups of steps, after warm-up, inputs resident), each in its own
    buffers, freed afterwards: the tiny step (also as 20 steps per CUDA
    graph), the GPT-2 124M step, the GPT-2 1.5B step without clip, the 7B
    all-reduce and the all-reduce sweep."""
    import torch
    import gradient_reduction_zero_gb300.dpz as dpz
    peak = peaks()["hbm_gbs"]
    rows = {}

    def row(w, ms, extra=None):
        b = step_bytes(w)
        r = {"ms_per_step": round(ms, 5), "value": round(b / (ms * 1e-3) / 1e9, 1), "unit": UNIT,
             "pct_of_measured_copy_peak": round(100 * b / (ms * 1e-3) / 1e9 / peak, 1),
             "steps_per_s": round(1e3 / ms, 1), "l2": l2_note(w)}
        if extra:
            r.update(extra)
        return r

    def zero1(w, steps):
        G, T, M, V, W = allocate(w, dev)
        ws = dpz.workspace(w.P, w.N, dev)
        nrm = torch.zeros(1, device=dev)
        cfg = dpz.make_cfg(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.step, w.clip)

        def step(on=stream):
            dpz.dp_zero1_step(G, T, M, V, W, w.N, cfg, ws=ws, norm_out=nrm, stream=on)
        warm_up(step, stream, max(3, args.warmup))
        ms = time_median(step, stream, steps)
        extra = {"clip": w.clip, "steps": steps}
        if w.P * w.N < 1 << 20:
            # launch-bound: the same steps through a prepared call (arguments
            # marshalled once), and the device time per step with 20 steps in
            # one graph
            call = dpz.prepare_zero1_step(G, T, M, V, W, w.N, cfg, ws=ws, norm_out=nrm,
                                          stream=stream)
            pms = time_median(call, stream, steps)
            extra.update(prepared_ms_per_step=round(pms, 5),
                         prepared_steps_per_s=round(1e3 / pms, 1))
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                on = torch.cuda.current_stream()
                for _ in range(20):
                    step(on)
            for _ in range(3):
                g.replay()
            gms = time_median(g.replay, torch.cuda.current_stream(), 100) / 20
            extra.update(graph_ms_per_step_20_per_graph=round(gms, 5),
                         graph_steps_per_s=round(1e3 / gms, 1))
        del G, T, M, V, W, ws
        torch.cuda.empty_cache()
        return row(w, ms, extra)

    def allreduce(w, steps):
        G, *_ = allocate(w, dev)
        warm_up(lambda: dpz.dp_allreduce_avg(G, w.N, stream), stream, max(3, args.warmup))
        ms = time_median(lambda: dpz.dp_allreduce_avg(G, w.N, stream), stream, steps)
        extra = {"steps": steps}
        if w.P * w.N < 1 << 20:
            call = dpz.prepare_allreduce_avg(G, w.N, stream=stream)
            pms = time_median(call, stream, steps)
            extra.update(prepared_ms_per_step=round(pms, 5),
                         prepared_steps_per_s=round(1e3 / pms, 1))
        del G
        torch.cuda.empty_cache()
        return row(w, ms, extra)

    rows[I.TINY.name] = zero1(I.TINY, 2000)
    rows[I.GPT2_124M.name] = zero1(I.GPT2_124M, 50)
    rows[I.GPT2_124M.name + " (no clip)"] = zero1(I.GPT2_124M.with_(clip=0.0), 50)
    rows[I.GPT2_1P5B.name + " (no clip)"] = zero1(I.GPT2_1P5B.with_(clip=0.0), 20)
    rows[I.ALLREDUCE_7B.name] = allreduce(I.ALLREDUCE_7B, 10)
    for n in (2, 4, 8):
        for size in I.SWEEP_SIZES:
            w = I.allreduce_sweep(size, n)
            rows[w.name] = allreduce(w, 200 if size < 1 << 26 else 20)
    return rows


def segment_bounds(P: int, N: int, k: int):
    """k buckets covering [0, P), bounds on 256-element segment boundaries of
    their chunks, in backward (last-first) order."""
    C = P // N
    edges = [0]
    for i in range(1, k):
        b = P * i // k
        c = b // C
        edges.append(c * C + (b - c * C) // 256 * 256)
    edges.append(P)
    edges = sorted(set(edges))
    return [(edges[i], edges[i + 1] - edges[i]) for i in range(len(edges) - 1)][::-1]


# The GEMM stand-in for a backward: bf16 matmuls of GEMM_DIM^3 (1.1 TFLOP each)
# per bucket.
GEMM_DIM = 8192
GEMM_PER_BUCKET = 3


def run_buckets(args, w, G, T, M, V, W, ws, nrm, cfg, stream, rs_ms):
    """Overlap of the reduce-scatter with a simulated backward pass.  The
    backward writes the gradient arena bucket by bucket (the seeded input
    generator, last bucket first) on the main stream.  Serial: the whole
    backward, then dp_zero1_step.  Overlapped: after each bucket an event;
    a second stream waits on it and reduces that bucket
    (dp_reduce_scatter_avg_range, capped at one block per SM so that the
    backward keeps most of the GPU), then finalises the norm and runs
    dp_zero1_update once the last bucket is in.  Both compute the same step.
    With --backward gemm each bucket's backward is instead GEMM_PER_BUCKET
    bf16 matmuls (the tensor cores, as a real backward's) followed by a copy
    of the bucket's gradients from a pre-generated arena."""
    import torch
    import gradient_reduction_zero_gb300.dpz as dpz
    es = w.grad_bytes()
    base = G.data_ptr()
    buckets = segment_bounds(w.P, w.N, args.buckets)
    main = stream
    # the reduction's blocks are dispatched ahead of the backward's as SMs free
    # up (the backward occupies every SM, as its GEMMs would)
    comm = torch.cuda.Stream(priority=-1)
    max_ctas = torch.cuda.get_device_properties(G.device).multi_processor_count

    if args.backward == "gemm":
        src = G.clone()                                  # the gradients the backward "produces"
        gen = torch.Generator(device=G.device).manual_seed(7)
        A = torch.randn(GEMM_DIM, GEMM_DIM, device=G.device, generator=gen).to(torch.bfloat16)
        B = torch.randn(GEMM_DIM, GEMM_DIM, device=G.device, generator=gen).to(torch.bfloat16)
        Cm = torch.empty(GEMM_DIM, GEMM_DIM, device=G.device, dtype=torch.bfloat16)
        Gv, Sv = G.view(w.N, w.P), src.view(w.N, w.P)

        def backward_bucket(lo, n):
            with torch.cuda.stream(main):
                for _ in range(GEMM_PER_BUCKET):
                    torch.matmul(A, B, out=Cm)
                Gv[:, lo:lo + n].copy_(Sv[:, lo:lo + n])
    else:
        def backward_bucket(lo, n):
            for r in range(w.N):
                I.dev_fill(base + (r * w.P + lo) * es, w.gdtype, lo, n, w.grad_seed + r,
                           I.STREAM_GRAD, w.grad, main.cuda_stream)

    def serial():
        for lo, n in buckets:
            backward_bucket(lo, n)
        dpz.dp_zero1_step(G, T, M, V, W, w.N, cfg, ws=ws, norm_out=nrm, stream=main)

    def overlapped():
        comm.wait_stream(main)
        for lo, n in buckets:
            backward_bucket(lo, n)
            ev = torch.cuda.Event()
            ev.record(main)
            comm.wait_event(ev)
            dpz.dp_reduce_scatter_avg_range(G, w.N, lo, n, ws=ws, stream=comm,
                                            max_ctas=max_ctas)
        dpz.dp_grad_norm_finalize(ws, w.P, w.N, nrm, stream=comm)
        dpz.dp_zero1_update(G, T, M, V, W, w.N, cfg, ws=ws, stream=comm)
        main.wait_stream(comm)

    def backward_only():
        for lo, n in buckets:
            backward_bucket(lo, n)

    def timed(fn, reps=3):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(main)
        for _ in range(reps):
            fn()
        e1.record(main)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    t_back = timed(backward_only)
    t_serial = timed(serial)
    t_over = timed(overlapped)
    # only the reduce-scatter can run before the last bucket exists; the norm
    # and the update need every bucket
    return {"buckets": len(buckets), "backward": args.backward, "max_ctas": max_ctas,
            "backward_ms": round(t_back, 3),
            "serial_ms": round(t_serial, 3), "overlapped_ms": round(t_over, 3),
            "reduce_scatter_ms": round(rs_ms, 3),
            "reduce_scatter_hidden_fraction": round((t_serial - t_over) / rs_ms, 3)}


def run_graph(args, step, stream, world, nbytes, per_graph=20):
    """The same step captured in a CUDA graph and replayed.  One step per
    graph is bounded by the host's launch of each replay; `per_graph` steps
    captured back to back in one graph give the device's time per step."""
    import torch

    def timed_graph(n_in_graph):
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            step_on = torch.cuda.current_stream()
            for _ in range(n_in_graph):
                step(step_on)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        reps = max(1, args.steps // n_in_graph)
        barrier(world)
        cur = torch.cuda.current_stream()
        e0.record(cur)
        for _ in range(reps):
            g.replay()
        e1.record(cur)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1) / (reps * n_in_graph), world)

    ms = timed_graph(1)
    ms_n = timed_graph(per_graph)
    return {"ms_per_step": round(ms, 5), "steps_per_s": round(1e3 / ms, 1),
            "value": round(nbytes * world / (ms * 1e-3) / 1e9, 2), "unit": UNIT,
            f"ms_per_step_{per_graph}_per_graph": round(ms_n, 5),
            f"steps_per_s_{per_graph}_per_graph": round(1e3 / ms_n, 1)}


def run_e2e(args, w, G, step_with, nrm, stream, world, full=None):
    """The step through the public API with the gradients coming from pinned
    host memory and the step's result (the norm; for an all-reduce one
    element) read back, every step.

    - Prefetched (the reported value unless --e2e-buckets is given): two
      gradient arenas; the host-to-device copy of step k+1's gradients runs on
      a copy stream while step k computes on the other arena, as a training
      loop prefetches its next batch.  Every step still copies its whole input
      and reads its result back; K steps are timed from the first copy to the
      last read, prologue and epilogue included.
    - Plain (always timed, reported as plain_ms_per_step): copy, then step.
    - --e2e-buckets K: within one step, the copy of bucket b (a copy engine,
      one stream) overlaps the reduce-scatter of bucket b-1
      (dp_reduce_scatter_avg_range on a second stream, ordered by an event
      per bucket); then the norm and the update."""
    import torch
    import gradient_reduction_zero_gb300.dpz as dpz
    host = torch.empty(G.shape, dtype=G.dtype, pin_memory=True)
    host.copy_(G)
    torch.cuda.synchronize()
    Gv, Hv = G.view(w.N, w.P), host.view(w.N, w.P)

    def result(buf):
        return nrm.item() if not w.allreduce_only else buf[:1].item()

    def plain():
        G.copy_(host, non_blocking=True)
        step_with(G, stream)
        return result(G)

    copy_s = torch.cuda.Stream()
    comm = torch.cuda.Stream(priority=-1)
    buckets = segment_bounds(w.P, w.N, args.e2e_buckets)[::-1]

    def pipelined():
        T, M, V, W, ws, cfg = full
        copy_s.wait_stream(stream)
        comm.wait_stream(stream)
        for lo, n in buckets:
            with torch.cuda.stream(copy_s):
                for r in range(w.N):          # one contiguous DMA copy per rank row
                    Gv[r, lo:lo + n].copy_(Hv[r, lo:lo + n], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(copy_s)
            comm.wait_event(ev)
            dpz.dp_reduce_scatter_avg_range(G, w.N, lo, n, ws=ws, stream=comm)
        dpz.dp_grad_norm_finalize(ws, w.P, w.N, nrm, stream=comm)
        dpz.dp_zero1_update(G, T, M, V, W, w.N, cfg, ws=ws, stream=comm)
        stream.wait_stream(comm)
        stream.wait_stream(copy_s)
        return nrm.item()

    def timed(fn):
        fn()
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            fn()
        torch.cuda.synchronize()
        return max_over_ranks((time.perf_counter() - t0) / args.e2e_steps, world)

    def prefetched_run(k):
        """k steps, double-buffered; returns seconds per step."""
        bufs = (G, G2)
        freed = [None, None]          # event: the last step that used the arena is done

        def copy_in(i):
            b = i % 2
            if freed[b] is not None:
                copy_s.wait_event(freed[b])
            with torch.cuda.stream(copy_s):
                bufs[b].copy_(host, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(copy_s)
            return ev

        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        ready = copy_in(0)
        for i in range(k):
            nxt = copy_in(i + 1) if i + 1 < k else None     # overlaps step i
            stream.wait_event(ready)
            step_with(bufs[i % 2], stream)
            done = torch.cuda.Event()
            done.record(stream)
            freed[i % 2] = done
            result(bufs[i % 2])                              # the read-back, every step
            ready = nxt
        torch.cuda.synchronize()
        return max_over_ranks((time.perf_counter() - t0) / k, world)

    dt_plain = timed(plain)
    use_pipe = full is not None and args.e2e_buckets > 1
    if use_pipe:
        dt = timed(pipelined)
        how = (f"pinned host gradients, {len(buckets)} buckets copied on one stream and "
               "reduced on another (dp_reduce_scatter_avg_range, events), then "
               "dp_grad_norm_finalize + dp_zero1_update; norm read back")
    else:
        G2 = torch.empty_like(G)
        prefetched_run(2)                                    # warm-up
        dt = prefetched_run(max(3, args.e2e_steps))
        del G2
        call = "dp_allreduce_avg" if w.allreduce_only else "dp_zero1_step"
        what = "one element" if w.allreduce_only else "the norm"
        how = (f"pinned host gradients copied on a copy stream into one of two arenas while "
               f"the previous step runs ({call}), {what} read back every step; "
               f"{max(3, args.e2e_steps)} steps timed from the first copy to the last read")
    d2h = 4 if not w.allreduce_only else G.element_size()
    out = {"value": round(step_bytes(w) * world / dt / 1e9, 2), "unit": UNIT,
           "ms_per_step": round(dt * 1e3, 3),
           "h2d_bytes_per_step": G.numel() * G.element_size(), "d2h_bytes_per_step": d2h,
           "how": how,
           "plain_ms_per_step": round(dt_plain * 1e3, 3)}
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["dpz", "reference"], default="dpz")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(I.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--e2e-buckets", type=int, default=0,
                    help="> 1: pipeline the e2e host copies with bucketed reduce-scatters")
    ap.add_argument("--entry", choices=ENTRIES, default="step",
                    help="time one entry point alone instead of the whole step")
    ap.add_argument("--clip", type=float, default=None,
                    help="override the workload's clip norm (0: no clipping, one fused kernel)")
    ap.add_argument("--buckets", type=int, default=0,
                    help="also measure a bucketed step overlapped with a simulated backward")
    ap.add_argument("--backward", choices=("fill", "gemm"), default="fill",
                    help="the simulated backward of --buckets: the seeded generator writing each "
                         "bucket (bound by instruction issue), or bf16 GEMMs on the tensor cores "
                         "followed by a copy of the bucket's gradients")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step captured in a CUDA graph and replayed")
    ap.add_argument("--acc32", action="store_true",
                    help="bf16 gradients reduced with fp32 accumulation (DPZ_BF16_ACC32)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads measured after the default one")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=4.0)
    args = ap.parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
