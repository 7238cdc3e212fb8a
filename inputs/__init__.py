"""Seeded synthetic inputs for the ZeRO-1 step: workload recipes and fillers.

This module makes input data only; it holds none of the step's arithmetic.
Both sides use it: the host build (``libinputs_host.so``) fills numpy arrays
for the CPU oracle, and the device build (``libinputs_dev.so``) fills the same
values into GPU memory.  ``gen.h`` defines the generator.

Workload recipes follow the pages' workloads (GPT-2 124M / 1.5B and a 7B
gradient arena, "A4 — Multi-GPU with NCCL and ZeRO-1"; "Lab 09 — Parallelism,
simulated" §1 and §4) as arena sizes and value distributions; no dataset or
checkpoint is involved.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(_HERE, "libinputs_host.so")
_DEV_SO = os.path.join(_HERE, "libinputs_dev.so")

ZERO, UNIFORM, NORMAL, NORMAL_TAIL, ABS_NORMAL = 0, 1, 2, 3, 4

# streams and seeds: rank r's gradients use seed (grad_seed + r)
STREAM_GRAD, STREAM_MASTER, STREAM_M, STREAM_V = 1, 2, 3, 4
SEED_MASTER, SEED_M, SEED_V = 1000, 1001, 1002


def _stale(target: str, sources: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def build_host() -> str:
    src = os.path.join(_HERE, "gen_host.c")
    hdr = os.path.join(_HERE, "gen.h")
    if _stale(_HOST_SO, [src, hdr]):
        tmp = _HOST_SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared",
                               "-ffp-contract=off", "-fno-fast-math",
                               src, "-o", tmp])
        os.replace(tmp, _HOST_SO)
    return _HOST_SO


def build_dev() -> str:
    src = os.path.join(_HERE, "gen_dev.cu")
    hdr = os.path.join(_HERE, "gen.h")
    if _stale(_DEV_SO, [src, hdr]):
        tmp = _DEV_SO + f".tmp{os.getpid()}"
        subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a",
                               "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                               "-fmad=false", src, "-o", tmp])
        os.replace(tmp, _DEV_SO)
    return _DEV_SO


_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        lib = ctypes.CDLL(build_host())
        for name, ptr in (("gen_fill_f32", ctypes.c_void_p), ("gen_fill_bf16", ctypes.c_void_p)):
            f = getattr(lib, name)
            f.argtypes = [ptr, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
                          ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_double]
            f.restype = None
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        lib = ctypes.CDLL(build_dev())
        for name in ("gen_fill_f32_dev", "gen_fill_bf16_dev"):
            f = getattr(lib, name)
            f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
                          ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                          ctypes.c_void_p]
            f.restype = ctypes.c_int
        _dev = lib
    return _dev


@dataclass(frozen=True)
class Dist:
    kind: int
    sigma: float = 0.0

    @property
    def scale(self) -> float:
        return self.sigma / 65536.0

    @property
    def scale_tail(self) -> float:
        return (self.sigma * 100.0) / 65536.0


@dataclass(frozen=True)
class Workload:
    """One synthetic ZeRO-1 (or ZeRO-0) step: sizes, dtypes, distributions and
    AdamW hyperparameters."""
    name: str
    N: int
    P: int
    gdtype: str = "bf16"          # "f32" | "bf16"
    wdtype: str = "bf16"
    grad: Dist = Dist(NORMAL, 1e-3)
    master: Dist = Dist(NORMAL, 0.02)
    m: Dist = Dist(ZERO)
    v: Dist = Dist(ZERO)
    grad_seed: int = 0
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.1
    step: int = 1
    clip: float = 0.0
    allreduce_only: bool = False  # ZeRO-0 all-reduce-average, no optimizer

    @property
    def C(self) -> int:
        return self.P // self.N

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    def grad_bytes(self) -> int:
        return 2 if self.gdtype == "bf16" else 4

    def weight_bytes(self) -> int:
        return 2 if self.wdtype == "bf16" else 4


def pad_params(P: int, N: int) -> int:
    """Zero-pad a parameter count to a multiple of 8*N (16-byte chunks)."""
    q = 8 * N
    return (P + q - 1) // q * q


# The five workloads.  Where a recipe leaves a value open, the choice is:
# master weights N(0, 0.02) everywhere; m = v = 0 and step 1 unless the recipe
# fixes them (the 1.5B recipe does); eps 1e-8; rank r's gradients seeded r.
TINY = Workload("tiny-zero1-n4-p4096", N=4, P=4096, gdtype="f32", wdtype="bf16",
                grad=Dist(UNIFORM), master=Dist(NORMAL, 0.02), lr=1e-3,
                beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1, step=1, clip=0.0)
GPT2_124M = Workload("gpt2-124m-zero1-n8", N=8, P=pad_params(124_439_808, 8),
                     grad=Dist(NORMAL, 1e-3), lr=6e-4, beta1=0.9, beta2=0.95,
                     eps=1e-8, weight_decay=0.1, step=1, clip=1.0)
GPT2_1P5B = Workload("gpt2-1.5b-zero1-n4", N=4, P=pad_params(1_557_611_200, 4),
                     grad=Dist(NORMAL_TAIL, 1e-3), m=Dist(NORMAL, 1e-4),
                     v=Dist(ABS_NORMAL, 1e-6), lr=1.5e-4, beta1=0.9, beta2=0.95,
                     eps=1e-8, weight_decay=0.1, step=1000, clip=1.0)


def allreduce_sweep(size_bytes: int, N: int) -> Workload:
    P = size_bytes // 4
    return Workload(f"allreduce-f32-{size_bytes}B-n{N}", N=N, P=P, gdtype="f32",
                    wdtype="f32", grad=Dist(UNIFORM), allreduce_only=True)


SWEEP_SIZES = [4096 * 4 ** k for k in range(10)]   # 4 KiB .. 1 GiB
ALLREDUCE_7B = Workload("allreduce-bf16-7b-n4", N=4, P=7_000_000_000, gdtype="bf16",
                        wdtype="bf16", grad=Dist(NORMAL, 1e-3), allreduce_only=True)

# The 1.5B workload's distributions on a 100M-parameter arena (2.8 GB resident,
# still far larger than L2): the case profiler captures run on.
PROFILE_1P5B_SHAPE = GPT2_1P5B.with_(name="zero1-n4-p100m-profile", P=100_000_000)

WORKLOADS = {w.name: w for w in (TINY, GPT2_124M, GPT2_1P5B, ALLREDUCE_7B, PROFILE_1P5B_SHAPE)}
WORKLOADS.update({w.name: w for w in (allreduce_sweep(s, n) for s in SWEEP_SIZES
                                      for n in (2, 4, 8))})


# ---------------------------------------------------------------- host fill

def _np_dtype(dt: str):
    return np.uint16 if dt == "bf16" else np.float32


def host_fill(dt: str, start: int, count: int, seed: int, stream: int, dist: Dist) -> np.ndarray:
    out = np.empty(count, dtype=_np_dtype(dt))
    if count:
        f = _host_lib().gen_fill_bf16 if dt == "bf16" else _host_lib().gen_fill_f32
        f(out.ctypes.data, start, count, seed, stream, dist.kind, dist.scale, dist.scale_tail)
    return out


def grads_host(w: Workload, rank: int, start: int = 0, count: int | None = None) -> np.ndarray:
    count = w.P - start if count is None else count
    return host_fill(w.gdtype, start, count, w.grad_seed + rank, STREAM_GRAD, w.grad)


def state_host(w: Workload, which: str, start: int = 0, count: int | None = None) -> np.ndarray:
    count = w.P - start if count is None else count
    d, seed, stream = {"master": (w.master, SEED_MASTER, STREAM_MASTER),
                       "m": (w.m, SEED_M, STREAM_M),
                       "v": (w.v, SEED_V, STREAM_V)}[which]
    return host_fill("f32", start, count, seed, stream, d)


def arena_host(w: Workload) -> np.ndarray:
    """grads[N][P] for a whole (small) workload."""
    return np.stack([grads_host(w, r) for r in range(w.N)])


def window_arena_host(w: Workload, offset: int, width: int) -> np.ndarray:
    """grads of a window: for every rank, elements [c*C + offset, +width) of
    every chunk c, laid out as a mini-arena [N][N*width] whose chunk c is the
    window of chunk c.  Element-wise results of the ring depend only on the
    chunk index, so a mini-arena checks the same elements."""
    C = w.C
    out = np.empty((w.N, w.N * width), dtype=_np_dtype(w.gdtype))
    for r in range(w.N):
        for c in range(w.N):
            out[r, c * width:(c + 1) * width] = grads_host(w, r, c * C + offset, width)
    return out


def window_state_host(w: Workload, which: str, offset: int, width: int) -> np.ndarray:
    C = w.C
    return np.concatenate([state_host(w, which, c * C + offset, width) for c in range(w.N)])


# ---------------------------------------------------------------- device fill

def dev_fill(ptr: int, dt: str, start: int, count: int, seed: int, stream_id: int,
             dist: Dist, cuda_stream: int = 0) -> None:
    lib = _dev_lib()
    f = lib.gen_fill_bf16_dev if dt == "bf16" else lib.gen_fill_f32_dev
    rc = f(ptr, start, count, seed, stream_id, dist.kind, dist.scale, dist.scale_tail,
           cuda_stream)
    if rc != 0:
        raise RuntimeError(f"device input generator failed (rc={rc})")


def fill_grads_device(w: Workload, grads, cuda_stream: int = 0) -> None:
    """grads: a contiguous device tensor holding N*P elements of w.gdtype."""
    es = w.grad_bytes()
    base = grads.data_ptr()
    for r in range(w.N):
        dev_fill(base + r * w.P * es, w.gdtype, 0, w.P, w.grad_seed + r, STREAM_GRAD,
                 w.grad, cuda_stream)


def fill_state_device(w: Workload, which: str, t, cuda_stream: int = 0) -> None:
    d, seed, stream = {"master": (w.master, SEED_MASTER, STREAM_MASTER),
                       "m": (w.m, SEED_M, STREAM_M),
                       "v": (w.v, SEED_V, STREAM_V)}[which]
    dev_fill(t.data_ptr(), "f32", 0, w.P, seed, stream, d, cuda_stream)
