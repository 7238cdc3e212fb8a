"""The timeout path of the bulk-copy staged kernels, on the GPU and without a
fault: a barrier that never completes (it expects 16 bytes more than the
kernel's loads deliver, and every load does complete) makes the bounded wait
run out.  The kernel sets the device flag, writes nothing and returns; the
host reads the flag through dpz_device_status, and the context stays usable."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import gradient_reduction_zero_gb300.dpz as dpz
    from gpu_util import DEV


def test_staged_wait_times_out_and_reports():
    assert dpz.device_status() == 0
    buf = torch.zeros(dpz.SELFTEST_BUF_BYTES // 4, dtype=torch.float32, device=DEV)
    buf[8:32] = 1.0                               # master, m, v of the one-tile arena
    before = buf.clone()
    try:
        t0 = time.perf_counter()
        dpz.selftest_staged_timeout(buf)
        torch.cuda.synchronize()
        waited = time.perf_counter() - t0
        assert dpz.device_status() == 1           # the bounded wait ran out
        assert dpz.device_status() == 0           # read and cleared
        assert torch.equal(buf, before)           # the abandoned tile wrote nothing
        assert 0.5 < waited < 60, waited
    finally:
        dpz.device_status()                       # never leave the flag set for later tests

    # the context is usable: a clipped step through the same kernel runs and
    # leaves the flag clear
    N, P = 4, 4 * 2048
    G = torch.randn(N * P, device=DEV).to(torch.bfloat16)
    T = torch.randn(P, device=DEV)
    M, V = torch.zeros_like(T), torch.zeros_like(T)
    W = torch.zeros(N * P, dtype=torch.bfloat16, device=DEV)
    ws = dpz.workspace(P, N, DEV)
    nrm = torch.zeros(1, device=DEV)
    cfg = dpz.make_cfg(1e-3, 0.9, 0.999, 1e-8, 0.1, 1, 1e-3)
    T0 = T.clone()
    dpz.dp_zero1_step(G, T, M, V, W, N, cfg, ws=ws, norm_out=nrm)
    torch.cuda.synchronize()
    assert dpz.device_status() == 0
    assert torch.isfinite(nrm).all() and nrm.item() > 0
    assert not torch.equal(T, T0)
    for r in range(1, N):
        assert torch.equal(W[r * P:(r + 1) * P], W[:P])
