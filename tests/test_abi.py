"""The C-ABI library without a GPU: it builds, loads, exports every symbol the
header declares, and rejects bad arguments before any CUDA call."""
import ctypes
import importlib.util
import os
import re
import subprocess
import sys

import pytest

from conftest import ROOT


def _build():
    path = os.path.join(ROOT, "gradient_reduction_zero_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("_dpz_build_t", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()


@pytest.fixture(scope="module")
def dpz():
    _build()
    import gradient_reduction_zero_gb300.dpz as d
    return d


def test_header_declares_the_step_calls(dpz):
    names = dpz.header_symbols()
    for n in ("dp_reduce_scatter_avg", "dp_allreduce_avg", "dp_grad_global_norm",
              "zero1_adamw_step", "dp_allgather", "dp_zero1_step", "dpz_workspace_bytes",
              "dpz_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(dpz):
    lib = ctypes.CDLL(dpz.LIB_PATH)
    names = dpz.header_symbols()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_bytes(dpz):
    # header + 256 first-stage sums + one double per 256-element segment
    segs = 4 * ((1_557_611_200 // 4 + 255) // 256)
    want = 256 + 8 * (256 + segs)
    assert dpz.lib.dpz_workspace_bytes(1_557_611_200, 4) == (want + 255) // 256 * 256
    assert dpz.lib.dpz_workspace_bytes(4096, 4) == (256 + 8 * (256 + 16) + 255) // 256 * 256
    assert dpz.lib.dpz_workspace_bytes(4098, 4) == 0
    assert dpz.lib.dpz_workspace_bytes(4096, 0) == 0


A = 0x7F0000000000          # fake, 16-byte aligned device addresses (never touched)
MB = 1 << 20


def _cfg(dpz, step=1, clip=0.0):
    return dpz.make_cfg(1e-3, 0.9, 0.999, 1e-8, 0.1, step, clip)


def _step(dpz, grads=A, master=A + 64 * MB, m=A + 80 * MB, v=A + 96 * MB,
          weights=A + 112 * MB, P=4096, N=4, g=0, w=1, cfg=None, ws=A + 200 * MB, norm=None):
    cfg = cfg or _cfg(dpz)
    return dpz.lib.dp_zero1_step(grads, master, m, v, weights, P, N, g, w, ctypes.byref(cfg),
                                 ws, norm, None)


@pytest.mark.parametrize("kw,code", [
    (dict(grads=None), 1),
    (dict(master=None), 1),
    (dict(weights=None), 1),
    (dict(N=0), 1),
    (dict(N=65), 1),
    (dict(P=0), 1),
    (dict(P=-8), 1),
    (dict(P=4098), 1),                  # P % N != 0
    (dict(P=4 * 1028), 2),              # chunk 1028 not a multiple of 8
    (dict(grads=A + 8), 2),             # misaligned
    (dict(m=A + 80 * MB + 4), 2),
    (dict(master=A + 64 * MB + 16), 2),  # fp32 buffers need 32-byte alignment
    (dict(g=0, grads=A + 16), 2),        # fp32 gradients too
    (dict(w=0, weights=A + 112 * MB + 16), 2),
    (dict(g=3), 1),                     # unknown dtype
    (dict(w=2), 1),                     # fp32 accumulation is a gradient mode only
    (dict(w=-1), 1),
    (dict(m=A + 64 * MB + 8192), 1),    # m overlaps master
    (dict(weights=A + 32 * 1024), 1),   # weights overlap grads (4*4096*4 bytes)
])
def test_zero1_step_rejects(dpz, kw, code):
    assert _step(dpz, **kw) == code
    assert dpz.lib.dpz_last_error().decode() != ""


def test_zero1_step_rejects_bad_step_and_missing_ws(dpz):
    assert _step(dpz, cfg=_cfg(dpz, step=0)) == 1
    assert b"step" in dpz.lib.dpz_last_error()
    # clipping needs the workspace
    assert _step(dpz, cfg=_cfg(dpz, clip=1.0), ws=None) == 1
    # ... but ws overlapping the weights is refused
    assert _step(dpz, cfg=_cfg(dpz, clip=1.0), ws=A + 112 * MB + 16) == 1


def test_other_calls_reject(dpz):
    L = dpz.lib
    assert L.dp_reduce_scatter_avg(None, 4096, 4, 0, None) == 1
    assert L.dp_reduce_scatter_avg(A, 4096, 4, 7, None) == 1
    assert L.dp_reduce_scatter_avg(A + 4, 4096, 4, 0, None) == 2
    assert L.dp_allreduce_avg(A, 4096, 3, 0, None) == 1          # 4096 % 3
    assert L.dp_allreduce_avg(A, 12, 3, 0, None) == 2            # chunk 4
    assert L.dp_allgather(A, 4096, 0, 1, None) == 1
    assert L.dp_grad_global_norm(A, 4096, 4, 1, None, None, None) == 1
    assert L.dp_grad_global_norm(A, 4096, 4, 1, A + 100, None, None) == 2
    assert L.dp_grad_global_norm(A, 4096, 4, 1, A + 64, None, None) == 1   # ws inside grads
    cfg = _cfg(dpz)
    assert L.zero1_adamw_step(A, None, A + MB, A + 2 * MB, A + 3 * MB, 4096, 4, 0, 0,
                              ctypes.byref(cfg), None, None) == 1
    assert L.zero1_adamw_step(A, A + MB, A + 2 * MB, A + 3 * MB, A + 4 * MB, 4096, 4, 0, 0,
                              None, None, None) == 1
    assert L.dpz_profile_start(0) == 1


def test_binding_fails_loudly_without_the_library(tmp_path):
    """The binding has no fallback: with libdpz.so absent, import raises."""
    pkg = tmp_path / "gradient_reduction_zero_gb300"
    pkg.mkdir()
    src = os.path.join(ROOT, "gradient_reduction_zero_gb300", "dpz.py")
    (pkg / "dpz.py").write_text(open(src).read())
    (pkg / "__init__.py").write_text("")
    code = ("import sys; sys.path.insert(0, %r)\n"
            "try:\n    import gradient_reduction_zero_gb300.dpz\n"
            "except ImportError as e:\n    print('raised', e)\n" % str(tmp_path))
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True)
    assert "raised" in out.stdout and "no CPU fallback" in out.stdout


def test_bucket_calls_reject(dpz):
    L = dpz.lib
    P, N = 4 * 6152, 4            # chunk 6152 = 24 segments of 256 + 8 elements
    ws = A + 512 * MB
    assert L.dp_reduce_scatter_avg_range(A, P, N, 1, -8, 64, None, 0, None) == 1
    assert L.dp_reduce_scatter_avg_range(A, P, N, 1, P - 8, 16, None, 0, None) == 1
    assert L.dp_reduce_scatter_avg_range(A, P, N, 1, 4, 64, None, 0, None) == 2      # lo % 8
    assert L.dp_reduce_scatter_avg_range(A, P, N, 1, 0, 12, None, 0, None) == 2      # n % 8
    # with norm partials the range must sit on segment boundaries of its chunks
    assert L.dp_reduce_scatter_avg_range(A, P, N, 1, 8, 256, ws, 0, None) == 2
    assert L.dp_reduce_scatter_avg_range(A, P, N, 1, 0, 6000, ws, 0, None) == 2
    assert L.dp_reduce_scatter_avg_range(A, P, N, 1, 0, 6152 + 256, A + 16, 0, None) == 1  # overlap
    # staging and shards must not overlap
    assert L.dp_reduce_scatter_avg_bucket(A, 0, 256, A + 512, P, N, 1, None, 0, None) == 1
    assert L.dp_reduce_scatter_avg_bucket(None, 0, 256, A + MB, P, N, 1, None, 0, None) == 1
    # a negative block cap
    assert L.dp_reduce_scatter_avg_range(A, P, N, 1, 0, 64, None, -1, None) == 1
    assert b"max_ctas" in L.dpz_last_error()
    assert L.dp_reduce_scatter_avg_bucket(A, 0, 256, A + MB, P, N, 1, None, -1, None) == 1
    assert L.dp_grad_norm_finalize(None, P, N, None, None) == 1
    cfg = _cfg(dpz, clip=1.0)
    assert L.dp_zero2_update(A, A + MB, A + 2 * MB, A + 3 * MB, A + 4 * MB, P, N, 1, 1,
                             ctypes.byref(cfg), None, None) == 1   # clip needs ws
    assert L.dp_zero1_update(A, A + MB + 16, A + 2 * MB, A + 3 * MB, A + 4 * MB, P, N, 1, 1,
                             ctypes.byref(_cfg(dpz)), None, None) == 2


def test_device_status_rejects_null(dpz):
    assert dpz.lib.dpz_device_status(None) == 1
    assert b"flag_out" in dpz.lib.dpz_last_error()


def test_selftest_rejects_bad_buffer(dpz):
    for k in (dpz.SELFTEST_UPDATE, dpz.SELFTEST_NORM, dpz.SELFTEST_STEP):
        assert dpz.lib.dpz_selftest_staged_timeout(k, None, None) == 1
        assert dpz.lib.dpz_selftest_staged_timeout(k, A + 16, None) == 2   # not 256-aligned
    assert dpz.lib.dpz_selftest_staged_timeout(3, A, None) == 1            # no such kernel
    assert b"kernel" in dpz.lib.dpz_last_error()


def test_header_constants_match_binding(dpz):
    """The status word's offset and bits, and the self-test's layout, as the
    header declares them."""
    text = open(dpz.HEADER).read()

    def define(name):
        m = re.search(r"#define\s+" + name + r"\s+(\d+)", text)
        assert m, name
        return int(m.group(1))

    assert define("DPZ_WS_STATUS_OFFSET") == dpz.WS_STATUS_OFFSET
    assert define("DPZ_STATUS_NORM_SKIPPED") == dpz.STATUS_NORM_SKIPPED
    assert define("DPZ_STATUS_UPDATE_SKIPPED") == dpz.STATUS_UPDATE_SKIPPED
    assert define("DPZ_SELFTEST_BUF_BYTES") == dpz.SELFTEST_BUF_BYTES
    assert [define(f"DPZ_SELFTEST_{k}") for k in ("UPDATE", "NORM", "STEP")] == \
        [dpz.SELFTEST_UPDATE, dpz.SELFTEST_NORM, dpz.SELFTEST_STEP]
    assert f"+{dpz.SELFTEST_NORM_OUT}  norm_out" in text
    assert f"+{dpz.SELFTEST_GRADS}  gradients" in text
    # the status word follows the header's double, float and three uint32
    assert dpz.WS_STATUS_OFFSET == 8 + 4 + 4 + 4
    # the self-test arena's workspace fits before norm_out
    assert dpz.lib.dpz_workspace_bytes(8, 1) <= dpz.SELFTEST_NORM_OUT


def test_division_selftest_rejects_bad_args(dpz):
    assert dpz.lib.dpz_selftest_average_division(0, A, None) == 1       # N < 1
    assert dpz.lib.dpz_selftest_average_division(65, A, None) == 1      # N > DPZ_MAX_RANKS
    assert dpz.lib.dpz_selftest_average_division(3, None, None) == 1    # NULL
    assert dpz.lib.dpz_selftest_average_division(3, A + 8, None) == 2   # misaligned
    assert b"mismatches" in dpz.lib.dpz_last_error()


def test_prepared_call_validates_every_call(dpz):
    """A prepared call makes the full C-ABI call each time, so the library's
    argument checks run on every call: a chunk that is not a whole number of
    8-element groups is refused before any launch (CPU tensors stand in for
    device memory; nothing is launched)."""
    import torch

    class NoStream:
        cuda_stream = 0

    N, P = 4, 4 * 12                        # chunk of 12 elements: not a multiple of 8
    G = torch.zeros(N * P)
    T, M, V = torch.zeros(P), torch.zeros(P), torch.zeros(P)
    W = torch.zeros(N * P, dtype=torch.bfloat16)
    cfg = dpz.make_cfg(1e-3, 0.9, 0.999, 1e-8, 0.1, 1)
    call = dpz.prepare_zero1_step(G, T, M, V, W, N, cfg, stream=NoStream())
    for _ in range(2):
        with pytest.raises(dpz.DpzError) as e:
            call()
        assert e.value.code == dpz.ERR_ALIGN
        assert "multiple of 8" in str(e.value)
    ar = dpz.prepare_allreduce_avg(G, N, stream=NoStream())
    with pytest.raises(dpz.DpzError):
        ar()


def test_call_module_covers_the_compute_calls(dpz):
    """The CPython call module (built where Python's headers are installed)
    exposes every compute call of the header with its arity, takes ints and
    None, and shares the one loaded libdpz.so with the ctypes binding: its
    errors read back through dpz_last_error."""
    if dpz._C is dpz.lib:
        pytest.skip("_dpzcall was not built here (no Python headers)")
    calls = {"dp_reduce_scatter_avg": 5, "dp_allreduce_avg": 5, "dp_grad_global_norm": 7,
             "dp_grad_global_norm_static": 6, "zero1_adamw_step": 12, "dp_allgather": 5,
             "dp_zero1_step": 13, "dp_reduce_scatter_avg_range": 9,
             "dp_reduce_scatter_avg_bucket": 10, "dp_grad_norm_finalize": 5,
             "dp_zero1_update": 12, "dp_zero2_update": 12}
    declared = set(dpz.header_symbols())
    for name, arity in calls.items():
        assert name in declared, name
        assert len(getattr(dpz.lib, name).argtypes) == arity, name
        fn = getattr(dpz._C, name)
        with pytest.raises(TypeError):
            fn(*([None] * (arity - 1)))
    # every compute call the header declares is in the module
    compute = {n for n in declared if n.startswith(("dp_", "zero1_"))}
    assert compute == set(calls)
    assert dpz._C.dp_allreduce_avg(None, 4096, 0, dpz.F32, None) == dpz.ERR_INVALID_ARG
    assert b"N = 0" in dpz.lib.dpz_last_error()
    assert dpz._C.dp_zero1_step(None, None, None, None, None, 4096, 4, dpz.F32, dpz.BF16,
                                None, None, None, None) == dpz.ERR_INVALID_ARG
    assert b"cfg is NULL" in dpz.lib.dpz_last_error()
    with pytest.raises(OverflowError):
        dpz._C.dp_allreduce_avg(None, 4096, 1 << 40, dpz.F32, None)
