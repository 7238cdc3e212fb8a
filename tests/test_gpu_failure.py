"""The timeout path of the bulk-copy staged kernels, on the GPU and without a
fault: a barrier that never completes (it expects 16 bytes more than the
kernel's loads deliver, and every load does complete) makes the bounded wait
run out, with a short bound so the test is quick.  The kernel gives up on its
tile and reports it twice: in stream order through the call's workspace (the
status word and a NaN norm in the workspace and in norm_out), and through the
device-wide flag that dpz_device_status reads.  It writes nothing of the
arena, and the context stays usable."""
import math
import time

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import gradient_reduction_zero_gb300.dpz as dpz
    from gpu_util import DEV


def _selftest_buffer():
    """The self-test buffer: a 256-byte aligned device tensor, the arena's
    gradients, master, m, v and weights filled with ones, norm_out = 5."""
    buf = torch.zeros(dpz.SELFTEST_BUF_BYTES // 4, dtype=torch.float32, device=DEV)
    assert buf.data_ptr() % 256 == 0
    b = buf.view(torch.uint8)
    g0 = dpz.SELFTEST_GRADS
    b[g0:g0 + 16].view(torch.bfloat16).fill_(1.0)              # gradients
    b[g0 + 32:g0 + 128].view(torch.float32).fill_(1.0)         # master, m, v
    b[g0 + 128:g0 + 144].view(torch.bfloat16).fill_(1.0)       # weights
    b[dpz.SELFTEST_NORM_OUT:dpz.SELFTEST_NORM_OUT + 4].view(torch.float32).fill_(5.0)
    return buf


@pytest.mark.parametrize("kernel,bits", [("UPDATE", 2), ("NORM", 1), ("STEP", 3)])
def test_staged_wait_times_out_and_reports(kernel, bits):
    assert dpz.device_status() == 0
    buf = _selftest_buffer()
    b = buf.view(torch.uint8)
    g0 = dpz.SELFTEST_GRADS
    arena_before = b[g0:g0 + 144].clone()
    try:
        t0 = time.perf_counter()
        dpz.selftest_staged_timeout(getattr(dpz, f"SELFTEST_{kernel}"), buf)
        torch.cuda.synchronize()
        waited = time.perf_counter() - t0
        assert dpz.device_status() == 1           # the bounded wait ran out
        assert dpz.device_status() == 0           # read and cleared
    finally:
        dpz.device_status()                       # never leave the flag set for later tests
    assert waited < 30, waited
    ws = b[:dpz.SELFTEST_NORM_OUT]
    assert dpz.ws_status(ws) == bits               # the call's own status word
    norm_out = b[dpz.SELFTEST_NORM_OUT:dpz.SELFTEST_NORM_OUT + 4].view(torch.float32).item()
    assert math.isnan(norm_out)                    # the norm the caller reads is NaN
    if kernel != "UPDATE":
        ws_norm = ws[8:12].view(torch.float32).item()
        assert math.isnan(ws_norm)                 # and so is the one in the workspace
    assert torch.equal(b[g0:g0 + 144], arena_before)   # the abandoned tile wrote nothing


def _step_inputs(N, P, seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    G = torch.randn(N * P, device=DEV, generator=gen).to(torch.bfloat16)
    T = torch.randn(P, device=DEV, generator=gen)
    return G, T, torch.zeros_like(T), torch.zeros_like(T), \
        torch.zeros(N * P, dtype=torch.bfloat16, device=DEV)


def test_context_usable_and_status_clear_after_timeouts():
    """After the self-tests a clipped step and a step without clip run, their
    workspaces' status words are 0 and the flag stays clear."""
    N, P = 4, 4 * 2048
    for clip in (1e-3, 0.0):
        G, T, M, V, W = _step_inputs(N, P, seed=3)
        ws = dpz.workspace(P, N, DEV)
        ws.fill_(0xFF)                             # a stale status word must be rewritten
        nrm = torch.zeros(1, device=DEV)
        cfg = dpz.make_cfg(1e-3, 0.9, 0.999, 1e-8, 0.1, 1, clip)
        T0 = T.clone()
        dpz.dp_zero1_step(G, T, M, V, W, N, cfg, ws=ws, norm_out=nrm)
        torch.cuda.synchronize()
        assert dpz.device_status() == 0
        assert dpz.ws_status(ws) == 0
        assert torch.isfinite(nrm).all() and nrm.item() > 0
        assert not torch.equal(T, T0)
        for r in range(1, N):
            assert torch.equal(W[r * P:(r + 1) * P], W[:P])


def test_update_with_skipped_norm_is_not_applied():
    """A clipped update whose norm's input was not read in full (status word
    NORM_SKIPPED, as the finalisation leaves it after a skipped tile) leaves
    master/m/v and the weights as they were and sets UPDATE_SKIPPED; both
    update kernels (the owner-only update and the update with the
    all-gather) do."""
    N, P = 4, 4 * 2048
    G, T, M, V, W = _step_inputs(N, P, seed=5)
    ws = dpz.workspace(P, N, DEV)
    dpz.dp_reduce_scatter_avg(G, N)
    dpz.dp_grad_global_norm(G, N, ws)
    torch.cuda.synchronize()
    assert dpz.ws_status(ws) == 0
    # what the finalisation writes when a tile of the norm was skipped
    ws[dpz.WS_STATUS_OFFSET:dpz.WS_STATUS_OFFSET + 4].view(torch.int32).fill_(
        dpz.STATUS_NORM_SKIPPED)
    ws[8:12].view(torch.float32).fill_(float("nan"))
    cfg = dpz.make_cfg(1e-3, 0.9, 0.999, 1e-8, 0.1, 1, 1.0)
    before = [t.clone() for t in (T, M, V, W)]
    for update in ("owner", "bcast"):
        if update == "owner":
            dpz.zero1_adamw_step(G, T, M, V, W, N, cfg, ws=ws)
        else:
            dpz.dp_zero1_update(G, T, M, V, W, N, cfg, ws=ws)
        torch.cuda.synchronize()
        assert dpz.ws_status(ws) == dpz.STATUS_NORM_SKIPPED | dpz.STATUS_UPDATE_SKIPPED
        for got, want in zip((T, M, V, W), before):
            assert torch.equal(got, want), update
        ws[dpz.WS_STATUS_OFFSET:dpz.WS_STATUS_OFFSET + 4].view(torch.int32).fill_(
            dpz.STATUS_NORM_SKIPPED)
    assert dpz.device_status() == 0
    # a fresh finalisation rewrites the word, and the update then runs
    dpz.dp_grad_global_norm(G, N, ws)
    dpz.dp_zero1_update(G, T, M, V, W, N, cfg, ws=ws)
    torch.cuda.synchronize()
    assert dpz.ws_status(ws) == 0
    assert not torch.equal(T, before[0])
    np.testing.assert_array_equal(W.view(N, P)[1].cpu().view(torch.int16).numpy(),
                                  W.view(N, P)[0].cpu().view(torch.int16).numpy())
