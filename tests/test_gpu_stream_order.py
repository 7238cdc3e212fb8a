"""Stream order with programmatic launches: every kernel of the library may be
placed on the GPU while the kernel before it on the stream still runs, and
must wait for it before touching memory.  These tests interleave library calls
with other kernels on one stream (torch copies that write the inputs, clones
that read the outputs) and chain library calls back to back, and require
every intermediate result to be the oracle's.  A kernel that read its inputs
before the previous kernel had written them, or wrote before the previous one
had read, would show as a wrong intermediate."""
import numpy as np
import pytest
import torch

import inputs as I
import oracle as O
from gpu_util import DEV, check_step, down, same_bits, up

pytestmark = pytest.mark.gpu


def _dpz():
    import gradient_reduction_zero_gb300.dpz as dpz
    return dpz


@pytest.mark.parametrize("N,C", [(4, 1024), (8, 12296)])
def test_allreduce_interleaved_with_other_kernels(N, C):
    """40 rounds of: a torch copy writes new inputs, the all-reduce, a torch
    clone reads the result; all queued on one stream before any check."""
    dpz = _dpz()
    P = N * C
    rng = np.random.default_rng(N * 1000 + C)
    srcs = [rng.uniform(-1, 1, (N, P)).astype(np.float32) for _ in range(40)]
    srcs_dev = [up(s) for s in srcs]
    G = torch.empty(N * P, dtype=torch.float32, device=DEV)
    outs = []
    for s in srcs_dev:
        G.copy_(s.view(-1))                  # another kernel writes the inputs
        dpz.dp_allreduce_avg(G, N)           # launched early, waits for the copy
        outs.append(G.clone())               # another kernel reads the result
    torch.cuda.synchronize()
    for s, o in zip(srcs, outs):
        ref = s.copy()
        O.ring_allreduce_avg(ref)
        assert same_bits(down(o).reshape(N, P), ref)


def test_chained_steps_with_reads_between():
    """30 ZeRO-1 steps (clip, N = 4) back to back on one stream, each followed
    by clones of the state and the weights and preceded by fresh gradients
    written by a torch copy, all queued before any check.  Each step must be
    the oracle's step applied to the state the GPU held before it."""
    dpz = _dpz()
    N, C = 4, 2056
    w = I.TINY.with_(N=N, P=N * C, gdtype="bf16", wdtype="bf16", clip=0.05,
                     grad=I.Dist(I.NORMAL, 1e-2), m=I.Dist(I.NORMAL, 1e-4),
                     v=I.Dist(I.ABS_NORMAL, 1e-6), step=10)
    th, m, v = (I.state_host(w, k) for k in ("master", "m", "v"))
    wts = np.zeros((N, w.P), dtype=np.uint16)
    grads = [I.arena_host(w.with_(grad_seed=100 + k)) for k in range(30)]
    T, M, V, W = up(th), up(m), up(v), up(wts)
    G = torch.empty(N * w.P, dtype=torch.bfloat16, device=DEV)
    ws = dpz.workspace(w.P, N, DEV)
    nrm = torch.zeros(1, device=DEV)
    gdev = [up(g) for g in grads]
    snaps = []
    for k in range(30):
        cfg = dpz.make_cfg(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.step + k, w.clip)
        G.copy_(gdev[k].view(-1))
        dpz.dp_zero1_step(G, T, M, V, W, N, cfg, ws=ws, norm_out=nrm)
        snaps.append((T.clone(), M.clone(), V.clone(), W.clone(), nrm.clone()))
    torch.cuda.synchronize()
    assert dpz.ws_status(ws) == 0
    prev = (th, m, v, wts)
    for k in range(30):
        Tg, Mg, Vg, Wg, ng = (down(x) for x in snaps[k])
        out = (None, Tg, Mg, Vg, Wg.reshape(N, w.P), float(ng[0]))
        check_step(w.with_(step=w.step + k), grads[k], *prev, out, check_avg=False)
        prev = (Tg, Mg, Vg, Wg.reshape(N, w.P))
