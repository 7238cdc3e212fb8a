"""dp_grad_global_norm_static: the global norm for callers that cannot
allocate device memory (for example a plug-in inside a framework whose caching
allocator owns the GPU, or a service that reserves its whole memory budget up
front).  It keeps its partial sums in a fixed 4 MiB device array that the
library declares, instead of a caller workspace.

The GPU test calls it through the C-ABI on arenas of different sizes and
seeds, two calls in a row in both orders (large then small, and small then
large, so that a slot or a first-stage sum left by a larger call would show),
and requires each result to equal, bit for bit, the workspace-based
dp_grad_global_norm (the same partials summed in the same fixed order), and
the oracle's norm within the relative 1e-6 of the other norm tests."""
import ctypes

import numpy as np
import pytest
import torch

import inputs as I

A = 0x7F0000000000      # a fake, aligned device address: never dereferenced


def _lib():
    import gradient_reduction_zero_gb300.dpz as dpz
    return dpz


def test_static_norm_rejects_arenas_beyond_its_scratch():
    """Sizes beyond the 4 MiB scratch are refused before any GPU work."""
    dpz = _lib()
    lib = dpz.lib
    # GPT-2 124M at N = 8 fits; the 1.5B arena at N = 4 does not
    assert dpz.lib.dpz_workspace_bytes(124_439_808, 8) <= 4 << 20
    rc = lib.dp_grad_global_norm_static(A, 1_557_611_200, 4, dpz.BF16, A - 64, None)
    assert rc == dpz.ERR_INVALID_ARG
    assert b"static scratch" in lib.dpz_last_error()
    rc = lib.dp_grad_global_norm_static(A, 4096, 4, dpz.BF16, None, None)
    assert rc == dpz.ERR_INVALID_ARG


def _oracle_norm(w):
    import oracle as O
    from oracle_windows import oracle_full_sumsq
    return O.clip_scale(oracle_full_sumsq(w), 0.0)[0]


@pytest.mark.gpu
@pytest.mark.parametrize("order", ["large-then-small", "small-then-large"])
def test_static_norm_matches_workspace_norm_twice(order):
    dpz = _lib()
    dev = torch.device("cuda:0")
    lib = ctypes.CDLL(dpz.LIB_PATH)
    fn = lib.dp_grad_global_norm_static
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                   ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    stream = torch.cuda.current_stream()
    # (N, C, gradient dtype, sigma, seed): the GPT-2 124M arena at N = 8, near
    # the scratch's limit, and a small fp32 arena at N = 3
    large = (8, 124_439_808 // 8, "bf16", 1e-3, 8)
    small = (3, 6152, "f32", 1.0, 3)
    cases = [large, small] if order == "large-then-small" else \
        [(3, 6152, "f32", 1.0, 31), (8, 124_439_808 // 8, "bf16", 1e-3, 81)]
    for N, C, gdt, sigma, seed in cases:
        w = I.TINY.with_(N=N, P=N * C, gdtype=gdt, grad=I.Dist(I.NORMAL, sigma), grad_seed=seed)
        G = torch.empty(w.N * w.P, dtype=torch.bfloat16 if gdt == "bf16" else torch.float32,
                        device=dev)
        I.fill_grads_device(w, G)
        dpz.dp_reduce_scatter_avg(G, N)               # owner chunks now hold the averages
        ws = dpz.workspace(w.P, N, dev)
        ref = torch.full((1,), -1.0, device=dev)
        dpz.dp_grad_global_norm(G, N, ws, ref)
        out = torch.full((1,), -2.0, device=dev)
        rc = fn(G.data_ptr(), w.P, N, dpz.BF16 if gdt == "bf16" else dpz.F32, out.data_ptr(),
                stream.cuda_stream)
        assert rc == 0, dpz.lib.dpz_last_error()
        torch.cuda.synchronize()
        r, o = ref.item(), out.item()
        assert np.float32(o).tobytes() == np.float32(r).tobytes(), (N, C, gdt, o, r)
        onorm = _oracle_norm(w)
        assert abs(o - onorm) <= 1e-6 * onorm, (N, C, gdt, o, onorm)
        assert dpz.ws_status(ws) == 0
        del G, ws
    torch.cuda.empty_cache()
    assert dpz.device_status() == 0
