"""Thin ctypes binding of libdpz.so (include/dpz.h): argument marshalling only.

Every function of the C-ABI is exposed under its own name.  Tensor arguments
are torch CUDA tensors (device memory and streams come from PyTorch); the
computation is entirely the library's own CUDA kernels.  If libdpz.so is
missing, importing this module raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdpz.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "dpz.h")

F32, BF16, BF16_ACC32 = 0, 1, 2
OK, ERR_INVALID_ARG, ERR_ALIGN, ERR_CUDA = 0, 1, 2, 3
MAX_RANKS = 64
# the per-call status word of a workspace (include/dpz.h)
WS_STATUS_OFFSET = 20
STATUS_NORM_SKIPPED, STATUS_UPDATE_SKIPPED = 1, 2


class DpzError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"dpz error {code}: {msg}")
        self.code = code


class AdamWCfg(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("step", ctypes.c_int64), ("clip_norm", ctypes.c_float),
                ("store_avg", ctypes.c_int)]


class KernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double)]


_VP = ctypes.c_void_p
_FP = ctypes.c_void_p     # float* (device)

_SIGS = {
    "dpz_workspace_bytes": ([ctypes.c_int64, ctypes.c_int], ctypes.c_size_t),
    "dp_reduce_scatter_avg": ([_VP, ctypes.c_int64, ctypes.c_int, ctypes.c_int, _VP], ctypes.c_int),
    "dp_allreduce_avg": ([_VP, ctypes.c_int64, ctypes.c_int, ctypes.c_int, _VP], ctypes.c_int),
    "dp_grad_global_norm": ([_VP, ctypes.c_int64, ctypes.c_int, ctypes.c_int, _VP, _FP, _VP],
                            ctypes.c_int),
    "zero1_adamw_step": ([_VP, _FP, _FP, _FP, _VP, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                          ctypes.c_int, _VP, _VP, _VP], ctypes.c_int),
    "dp_allgather": ([_VP, ctypes.c_int64, ctypes.c_int, ctypes.c_int, _VP], ctypes.c_int),
    "dp_zero1_step": ([_VP, _FP, _FP, _FP, _VP, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                       ctypes.c_int, _VP, _VP, _FP, _VP], ctypes.c_int),
    "dp_grad_global_norm_static": ([_VP, ctypes.c_int64, ctypes.c_int, ctypes.c_int, _FP, _VP],
                                   ctypes.c_int),
    "dp_reduce_scatter_avg_range": ([_VP, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int64, ctypes.c_int64, _VP, ctypes.c_int, _VP],
                                    ctypes.c_int),
    "dp_reduce_scatter_avg_bucket": ([_VP, ctypes.c_int64, ctypes.c_int64, _VP, ctypes.c_int64,
                                      ctypes.c_int, ctypes.c_int, _VP, ctypes.c_int, _VP],
                                     ctypes.c_int),
    "dp_grad_norm_finalize": ([_VP, ctypes.c_int64, ctypes.c_int, _FP, _VP], ctypes.c_int),
    "dp_zero1_update": ([_VP, _FP, _FP, _FP, _VP, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                         ctypes.c_int, _VP, _VP, _VP], ctypes.c_int),
    "dp_zero2_update": ([_VP, _FP, _FP, _FP, _VP, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                         ctypes.c_int, _VP, _VP, _VP], ctypes.c_int),
    "dpz_last_error": ([], ctypes.c_char_p),
    "dpz_version": ([], ctypes.c_char_p),
    "dpz_launch_count": ([], ctypes.c_int64),
    "dpz_device_status": ([ctypes.POINTER(ctypes.c_int)], ctypes.c_int),
    "dpz_selftest_staged_timeout": ([ctypes.c_int, _VP, _VP], ctypes.c_int),
    "dpz_selftest_average_division": ([ctypes.c_int, _VP, _VP], ctypes.c_int),
    "dpz_profile_start": ([ctypes.c_int], ctypes.c_int),
    "dpz_profile_stop": ([ctypes.POINTER(KernelStat), ctypes.c_int,
                          ctypes.POINTER(ctypes.c_int)], ctypes.c_int),
}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run gradient_reduction_zero_gb300.build.build() "
            "(there is no CPU fallback)")
    L = ctypes.CDLL(LIB_PATH)
    for name, (args, res) in _SIGS.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    return L


lib = _load()


def _load_call():
    """The CPython module that makes the compute calls (loaded after lib, so
    that both use the one loaded libdpz.so); lib itself where it was not
    built.  Both take the same arguments: Python ints, None for NULL."""
    try:
        from . import _dpzcall
    except ImportError:
        return lib
    return _dpzcall


_C = _load_call()


def header_symbols(path: str = HEADER) -> list[str]:
    """Names of the functions include/dpz.h declares."""
    text = open(path).read()
    return re.findall(r"DPZ_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def _check(rc: int) -> None:
    if rc != OK:
        raise DpzError(rc, lib.dpz_last_error().decode())


# ------------------------------------------------------------ tensor helpers

def _torch():
    import torch
    return torch


_CODES: dict = {}


def dtype_code(t, acc32: bool = False) -> int:
    """DPZ dtype code of a tensor; acc32 selects the fp32-accumulating ring for
    a bf16 gradient arena."""
    if not _CODES:
        torch = _torch()
        _CODES.update({torch.bfloat16: BF16, torch.float32: F32})
    code = _CODES.get(t.dtype)
    if code is None:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if acc32:
        if code != BF16:
            raise TypeError("fp32 accumulation applies to bf16 gradient arenas")
        return BF16_ACC32
    return code


def _stream_handle(stream) -> int:
    if stream is None:
        stream = _torch().cuda.current_stream()
    return stream.cuda_stream


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def make_cfg(lr, beta1, beta2, eps, weight_decay, step, clip_norm=0.0, store_avg=False) -> AdamWCfg:
    return AdamWCfg(lr, beta1, beta2, eps, weight_decay, int(step), clip_norm, int(bool(store_avg)))


def workspace(P: int, N: int, device=None):
    """A device tensor of dpz_workspace_bytes(P, N) bytes."""
    torch = _torch()
    nb = lib.dpz_workspace_bytes(P, N)
    if nb == 0:
        raise DpzError(ERR_INVALID_ARG, f"no workspace size for P={P}, N={N}")
    return torch.empty(nb, dtype=torch.uint8, device=device or "cuda")


def _np(arena, N: int) -> int:
    n = arena.numel()
    if n % N:
        raise ValueError("arena size is not a multiple of N")
    return n // N


# ------------------------------------------------------------ the calls

def dp_reduce_scatter_avg(grads, N: int, stream=None, acc32: bool = False) -> None:
    _check(_C.dp_reduce_scatter_avg(_ptr(grads), _np(grads, N), N, dtype_code(grads, acc32),
                                     _stream_handle(stream)))


def dp_allreduce_avg(grads, N: int, stream=None, acc32: bool = False) -> None:
    _check(_C.dp_allreduce_avg(_ptr(grads), _np(grads, N), N, dtype_code(grads, acc32),
                                _stream_handle(stream)))


def dp_grad_global_norm(grads, N: int, ws, norm_out=None, stream=None) -> None:
    _check(_C.dp_grad_global_norm(_ptr(grads), _np(grads, N), N, dtype_code(grads), _ptr(ws),
                                   _ptr(norm_out), _stream_handle(stream)))


def dp_grad_global_norm_static(grads, N: int, norm_out, stream=None) -> None:
    """The global norm without a caller workspace (fixed device scratch)."""
    _check(_C.dp_grad_global_norm_static(_ptr(grads), _np(grads, N), N, dtype_code(grads),
                                          _ptr(norm_out), _stream_handle(stream)))


def zero1_adamw_step(grads, master, m, v, weights, N: int, cfg: AdamWCfg, ws=None,
                     stream=None) -> None:
    _check(_C.zero1_adamw_step(_ptr(grads), _ptr(master), _ptr(m), _ptr(v), _ptr(weights),
                                _np(grads, N), N, dtype_code(grads), dtype_code(weights),
                                ctypes.addressof(cfg), _ptr(ws), _stream_handle(stream)))


def dp_allgather(weights, N: int, stream=None) -> None:
    _check(_C.dp_allgather(_ptr(weights), _np(weights, N), N, dtype_code(weights),
                            _stream_handle(stream)))


def dp_zero1_step(grads, master, m, v, weights, N: int, cfg: AdamWCfg, ws=None, norm_out=None,
                  stream=None, acc32: bool = False) -> None:
    _check(_C.dp_zero1_step(_ptr(grads), _ptr(master), _ptr(m), _ptr(v), _ptr(weights),
                             _np(grads, N), N, dtype_code(grads, acc32), dtype_code(weights),
                             ctypes.addressof(cfg), _ptr(ws), _ptr(norm_out),
                             _stream_handle(stream)))


def dp_reduce_scatter_avg_range(grads, N: int, lo: int, n: int, ws=None, stream=None,
                                acc32: bool = False, max_ctas: int = 0) -> None:
    """max_ctas: 0 = one pass over the range; > 0 caps the kernel's blocks
    (for example one per SM) to leave the GPU to kernels on other streams."""
    _check(_C.dp_reduce_scatter_avg_range(_ptr(grads), _np(grads, N), N, dtype_code(grads, acc32),
                                           lo, n, _ptr(ws), max_ctas, _stream_handle(stream)))


def dp_reduce_scatter_avg_bucket(staging, lo: int, shards, N: int, ws=None, stream=None,
                                 acc32: bool = False, max_ctas: int = 0) -> None:
    """staging: [N*n] (rank r's values of arena elements [lo, lo+n) at r*n);
    shards: [P].  max_ctas as in dp_reduce_scatter_avg_range."""
    n = _np(staging, N)
    _check(_C.dp_reduce_scatter_avg_bucket(_ptr(staging), lo, n, _ptr(shards), shards.numel(),
                                            N, dtype_code(staging, acc32), _ptr(ws), max_ctas,
                                            _stream_handle(stream)))


def dp_grad_norm_finalize(ws, P: int, N: int, norm_out=None, stream=None) -> None:
    _check(_C.dp_grad_norm_finalize(_ptr(ws), P, N, _ptr(norm_out), _stream_handle(stream)))


def dp_zero1_update(grads, master, m, v, weights, N: int, cfg: AdamWCfg, ws=None,
                    stream=None) -> None:
    _check(_C.dp_zero1_update(_ptr(grads), _ptr(master), _ptr(m), _ptr(v), _ptr(weights),
                               _np(grads, N), N, dtype_code(grads), dtype_code(weights),
                               ctypes.addressof(cfg), _ptr(ws), _stream_handle(stream)))


def dp_zero2_update(shards, master, m, v, weights, N: int, cfg: AdamWCfg, ws=None,
                    stream=None) -> None:
    _check(_C.dp_zero2_update(_ptr(shards), _ptr(master), _ptr(m), _ptr(v), _ptr(weights),
                               shards.numel(), N, dtype_code(shards), dtype_code(weights),
                               ctypes.addressof(cfg), _ptr(ws), _stream_handle(stream)))


class PreparedCall:
    """One C-ABI call whose arguments were marshalled once: calling it makes
    the same call again (the library validates the arguments and launches its
    kernels every time).  For a training loop that runs the same step on the
    same buffers, this leaves out the per-call Python work of turning tensors
    into pointers and dtype codes.  It keeps the tensors and the AdamW
    settings alive; changing a cfg field after preparing changes the calls."""
    __slots__ = ("_fn", "_args", "_keep")

    def __init__(self, fn, args, keep):
        self._fn = fn
        self._args = tuple(args)
        self._keep = keep

    def __call__(self) -> None:
        rc = self._fn(*self._args)
        if rc != OK:
            _check(rc)


def _prepare(name: str, args: tuple, keep) -> PreparedCall:
    """A PreparedCall of the compute call `name` with `args` (Python ints,
    None for NULL).  Through ctypes they are converted here, once."""
    fn = getattr(_C, name)
    if _C is lib:
        args = tuple(t(v) for t, v in zip(fn.argtypes, args))
    return PreparedCall(fn, args, keep)


def prepare_zero1_step(grads, master, m, v, weights, N: int, cfg: AdamWCfg, ws=None,
                       norm_out=None, stream=None, acc32: bool = False) -> PreparedCall:
    """dp_zero1_step with its arguments marshalled once (PreparedCall)."""
    args = (_ptr(grads), _ptr(master), _ptr(m), _ptr(v), _ptr(weights), _np(grads, N), N,
            dtype_code(grads, acc32), dtype_code(weights), ctypes.addressof(cfg), _ptr(ws),
            _ptr(norm_out), _stream_handle(stream))
    return _prepare("dp_zero1_step", args, (grads, master, m, v, weights, cfg, ws, norm_out))


def prepare_allreduce_avg(grads, N: int, stream=None, acc32: bool = False) -> PreparedCall:
    """dp_allreduce_avg with its arguments marshalled once (PreparedCall)."""
    args = (_ptr(grads), _np(grads, N), N, dtype_code(grads, acc32), _stream_handle(stream))
    return _prepare("dp_allreduce_avg", args, (grads,))


def launch_count() -> int:
    return int(lib.dpz_launch_count())


def device_status() -> int:
    """The device error flag (1 if a kernel's bounded wait on its own copies
    ran out since the last call), read and cleared."""
    f = ctypes.c_int()
    _check(lib.dpz_device_status(ctypes.byref(f)))
    return f.value


def ws_status(ws) -> int:
    """The DPZ_STATUS_* bits of a workspace tensor's status word (a read of
    device memory; it synchronises with the current stream)."""
    return int(ws[WS_STATUS_OFFSET:WS_STATUS_OFFSET + 4].view(_torch().int32).item())


SELFTEST_BUF_BYTES = 4096
SELFTEST_UPDATE, SELFTEST_NORM, SELFTEST_STEP = 0, 1, 2
# offsets in the self-test buffer (include/dpz.h)
SELFTEST_NORM_OUT, SELFTEST_GRADS = 2560, 2816


def selftest_staged_timeout(kernel: int, buf, stream=None) -> None:
    """Launch one staged kernel (SELFTEST_*) on the one-tile arena laid out in
    `buf` (a 256-byte aligned device tensor of at least SELFTEST_BUF_BYTES
    bytes) with a barrier that never completes and a short wait bound, so
    that the kernel gives up on its tile and reports it."""
    if buf.numel() * buf.element_size() < SELFTEST_BUF_BYTES:
        raise ValueError(f"buf must hold at least {SELFTEST_BUF_BYTES} bytes")
    _check(lib.dpz_selftest_staged_timeout(int(kernel), _ptr(buf), _stream_handle(stream)))


def selftest_average_division(N: int, counter, stream=None) -> None:
    """Count, into `counter` (a device int64 tensor of one element), the
    float inputs whose average division by N differs bit for bit from an
    IEEE division, over all 2^32 bit patterns; 0 means correctly rounded."""
    if counter.numel() != 1 or counter.element_size() != 8:
        raise ValueError("counter must be a one-element 8-byte tensor")
    _check(lib.dpz_selftest_average_division(int(N), _ptr(counter), _stream_handle(stream)))


def version() -> str:
    return lib.dpz_version().decode()


def profile_start(max_launches: int = 4096) -> None:
    _check(lib.dpz_profile_start(max_launches))


def profile_stop() -> dict:
    """{kernel name: (launches, total_ms)} for the launches since profile_start."""
    stats = (KernelStat * 64)()
    n = ctypes.c_int()
    _check(lib.dpz_profile_stop(stats, 64, ctypes.byref(n)))
    return {stats[i].name.decode(): (int(stats[i].launches), float(stats[i].total_ms))
            for i in range(min(n.value, 64))}
