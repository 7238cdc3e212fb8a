"""CPU oracle for the data-parallel / ZeRO-1 step (ctypes wrapper of oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg may call it; the product path never does.  It shares no code
with the CUDA library.  Arrays: float64 -> F64, float32 -> F32, uint16 -> bf16
bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
# a test may point the wrapper at another build of oracle.c (a planted mistake)
_OVERRIDE = os.environ.get("DPZ_ORACLE_LIB")

F32, BF16, F64, BF16_ACC32 = 0, 1, 2, 3


def build() -> str:
    if _OVERRIDE:
        return _OVERRIDE
    src = os.path.join(_HERE, "oracle.c")
    hdr = os.path.join(_HERE, "oracle.h")
    if (not os.path.exists(_SO) or os.path.getmtime(src) > os.path.getmtime(_SO)
            or os.path.getmtime(hdr) > os.path.getmtime(_SO)):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off",
                               "-fno-fast-math", "-fPIC", "-shared", src, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class AdamWCfg(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("eps", ctypes.c_float),
                ("weight_decay", ctypes.c_float), ("step", ctypes.c_int64),
                ("clip_norm", ctypes.c_float)]


_lib = None
_P = ctypes.c_void_p
_I64P = ctypes.POINTER(ctypes.c_int64)


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        sig = {
            "orc_f32_to_bf16": ([ctypes.c_float], ctypes.c_uint16),
            "orc_bf16_to_f32": ([ctypes.c_uint16], ctypes.c_float),
            "orc_f32_to_bf16_array": ([_P, _P, ctypes.c_int64], None),
            "orc_ring_reduce_scatter": ([_P, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, _P], ctypes.c_int),
            "orc_ring_allgather": ([_P, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, _P], ctypes.c_int),
            "orc_owner": ([ctypes.c_int, ctypes.c_int, ctypes.c_int], ctypes.c_int),
            "orc_average_owned": ([_P, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                   ctypes.c_int], ctypes.c_int),
            "orc_ring_allreduce_avg": ([_P, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                        ctypes.c_int, _P], ctypes.c_int),
            "orc_reduce_scatter_avg": ([_P, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                        ctypes.c_int, _P], ctypes.c_int),
            "orc_star_allreduce": ([_P, ctypes.c_int, ctypes.c_int64, ctypes.c_int, _P],
                                   ctypes.c_int),
            "orc_sumsq_owned": ([_P, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int],
                                ctypes.c_double),
            "orc_clip_scale": ([ctypes.c_double, ctypes.c_float, _P, _P], None),
            "orc_adamw": ([_P, _P, _P, _P, ctypes.c_int, ctypes.c_int64,
                           ctypes.POINTER(AdamWCfg), ctypes.c_float], None),
            "orc_bias_corrections": ([ctypes.POINTER(AdamWCfg), _P, _P], None),
            "orc_zero1_step": ([_P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                ctypes.c_int, ctypes.POINTER(AdamWCfg), ctypes.c_double,
                                _P, _P, _P, _P], ctypes.c_int),
            "orc_zero0_step": ([_P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                ctypes.c_int, ctypes.POINTER(AdamWCfg), _P, _P], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"unsupported oracle dtype {a.dtype}")


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


def _chk(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments")


def cfg_of(lr, beta1, beta2, eps, weight_decay, step, clip_norm=0.0) -> AdamWCfg:
    return AdamWCfg(lr, beta1, beta2, eps, weight_decay, int(step), clip_norm)


def cfg_from_workload(w) -> AdamWCfg:
    return cfg_of(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.step, w.clip)


# ------------------------------------------------------------------ wrappers

def f32_to_bf16(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f32_to_bf16_array(_ptr(x), _ptr(out), x.size)
    return out


def bf16_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def _code(arena: np.ndarray, acc32: bool) -> int:
    if acc32:
        if arena.dtype != np.uint16:
            raise TypeError("fp32 accumulation applies to bf16 arenas")
        return BF16_ACC32
    return dtype_code(arena)


def ring_reduce_scatter(arena: np.ndarray, rho: int = 1, steps: int | None = None,
                        acc32: bool = False):
    """In place on arena[N][P]; returns bytes sent per rank.  acc32: a bf16
    arena whose ring carries fp32 partial sums."""
    N, P = arena.shape
    steps = N - 1 if steps is None else steps
    sent = np.zeros(N, dtype=np.int64)
    _chk(lib().orc_ring_reduce_scatter(_ptr(arena), N, P, _code(arena, acc32), rho, steps,
                                       _ptr(sent)), "reduce-scatter")
    return sent


def ring_allgather(arena: np.ndarray, rho: int = 1, steps: int | None = None):
    N, P = arena.shape
    steps = N - 1 if steps is None else steps
    sent = np.zeros(N, dtype=np.int64)
    _chk(lib().orc_ring_allgather(_ptr(arena), N, P, dtype_code(arena), rho, steps,
                                  _ptr(sent)), "all-gather")
    return sent


def owner(c: int, N: int, rho: int = 1) -> int:
    return lib().orc_owner(c, N, rho)


def average_owned(arena: np.ndarray, rho: int = 1) -> None:
    N, P = arena.shape
    _chk(lib().orc_average_owned(_ptr(arena), N, P, dtype_code(arena), rho), "average")


def reduce_scatter_avg(arena: np.ndarray, rho: int = 1, acc32: bool = False):
    """Reduce-scatter then owner average in one ring session (needed for acc32,
    whose fp32 partial sums exist only inside the ring).  In place; only the
    owner chunks are meaningful afterwards.  Returns bytes sent per rank."""
    N, P = arena.shape
    sent = np.zeros(N, dtype=np.int64)
    _chk(lib().orc_reduce_scatter_avg(_ptr(arena), N, P, _code(arena, acc32), rho, _ptr(sent)),
         "reduce-scatter")
    return sent


def ring_allreduce_avg(arena: np.ndarray, rho: int = 1, acc32: bool = False):
    N, P = arena.shape
    sent = np.zeros(N, dtype=np.int64)
    _chk(lib().orc_ring_allreduce_avg(_ptr(arena), N, P, _code(arena, acc32), rho,
                                      _ptr(sent)), "all-reduce")
    return sent


def star_allreduce(arena: np.ndarray):
    N, P = arena.shape
    recv = np.zeros(N, dtype=np.int64)
    _chk(lib().orc_star_allreduce(_ptr(arena), N, P, dtype_code(arena), _ptr(recv)), "star")
    return recv


def sumsq_owned(arena: np.ndarray, rho: int = 1) -> float:
    N, P = arena.shape
    return lib().orc_sumsq_owned(_ptr(arena), N, P, dtype_code(arena), rho)


def clip_scale(sumsq: float, clip: float):
    n = ctypes.c_float()
    s = ctypes.c_float()
    lib().orc_clip_scale(sumsq, clip, ctypes.addressof(n), ctypes.addressof(s))
    return n.value, s.value


def bias_corrections(cfg: AdamWCfg):
    b1 = ctypes.c_float()
    b2 = ctypes.c_float()
    lib().orc_bias_corrections(ctypes.byref(cfg), ctypes.addressof(b1), ctypes.addressof(b2))
    return b1.value, b2.value


def adamw(theta, m, v, grad, cfg: AdamWCfg, scale: float = 1.0) -> None:
    """In place on float32 theta/m/v; grad float32 or bf16 (uint16)."""
    n = theta.size
    assert m.size == n and v.size == n and grad.size == n
    lib().orc_adamw(_ptr(theta), _ptr(m), _ptr(v), _ptr(grad), dtype_code(grad), n,
                    ctypes.byref(cfg), scale)


def zero1_step(grads, master, m, v, weights, cfg: AdamWCfg, ext_sumsq: float = -1.0,
               acc32: bool = False):
    """In place.  Returns (norm, scale, sent_rs, sent_ag)."""
    N, P = grads.shape
    assert weights.shape == (N, P)
    norm = ctypes.c_float()
    scale = ctypes.c_float()
    srs = np.zeros(N, dtype=np.int64)
    sag = np.zeros(N, dtype=np.int64)
    _chk(lib().orc_zero1_step(_ptr(grads), _ptr(master), _ptr(m), _ptr(v), _ptr(weights),
                              N, P, _code(grads, acc32), dtype_code(weights), ctypes.byref(cfg),
                              ext_sumsq, ctypes.addressof(norm), ctypes.addressof(scale),
                              _ptr(srs), _ptr(sag)), "zero1 step")
    return norm.value, scale.value, srs, sag


def zero0_step(grads, master_full, m_full, v_full, weights, cfg: AdamWCfg):
    """In place; master_full/m_full/v_full are [N][P].  Returns (norm, sent)."""
    N, P = grads.shape
    norm = ctypes.c_float()
    sent = np.zeros(N, dtype=np.int64)
    _chk(lib().orc_zero0_step(_ptr(grads), _ptr(master_full), _ptr(m_full), _ptr(v_full),
                              _ptr(weights), N, P, dtype_code(grads), dtype_code(weights),
                              ctypes.byref(cfg), ctypes.addressof(norm), _ptr(sent)),
         "zero0 step")
    return norm.value, sent
