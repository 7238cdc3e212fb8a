"""Guard bands around every buffer of every entry point: each call runs on
views into larger allocations whose bytes before and after the view hold
canary values, and no canary may change.  A kernel that wrote one element past
a chunk, a ragged segment or a workspace would show here, where the parity
tests (which compare only the buffers' own elements) could not see it.

Two arenas, N = 4: chunks of 2,056 elements span several 1024-element tiles
and 256-element segments; chunks of 1,032 (20 segments in all) take the
small-arena step.  Both end every chunk with a ragged segment of 8."""
import numpy as np
import pytest
import torch

import inputs as I

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
PAD = 4096                 # bytes of guard band on each side (keeps 256-byte alignment)
N = 4


def _dpz():
    import gradient_reduction_zero_gb300.dpz as dpz
    return dpz


class Guarded:
    """A tensor of `numel` elements of `dtype` inside guard bands of PAD bytes
    that hold the byte 0xA5."""

    def __init__(self, numel, dtype):
        es = torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((numel * es + 2 * PAD,), 0xA5, dtype=torch.uint8, device=DEV)
        self.view = self.raw[PAD:PAD + numel * es].view(dtype)

    def intact(self):
        head, tail = self.raw[:PAD], self.raw[-PAD:]
        return bool((head == 0xA5).all()) and bool((tail == 0xA5).all())


def _problem(C, gdt, wdt):
    P = N * C
    w = I.TINY.with_(N=N, P=P, gdtype=gdt, wdtype=wdt, grad=I.Dist(I.NORMAL, 1e-2),
                     m=I.Dist(I.NORMAL, 1e-4), v=I.Dist(I.ABS_NORMAL, 1e-6), step=10)
    gt = torch.bfloat16 if gdt == "bf16" else torch.float32
    wt = torch.bfloat16 if wdt == "bf16" else torch.float32
    G = Guarded(N * P, gt)
    I.fill_grads_device(w, G.view)
    T, M, V = (Guarded(P, torch.float32) for _ in range(3))
    for k, t in (("master", T), ("m", M), ("v", V)):
        I.fill_state_device(w, k, t.view)
    W = Guarded(N * P, wt)
    W.view.zero_()
    ws = Guarded(_dpz().lib.dpz_workspace_bytes(P, N), torch.uint8)
    ws.view.zero_()
    nrm = Guarded(1, torch.float32)
    cfg = _dpz().make_cfg(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.step, 0.05)
    return G, T, M, V, W, ws, nrm, cfg


def _no_clip(cfg):
    return _dpz().make_cfg(cfg.lr, cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay, cfg.step, 0.0)


def _entry(name, C, G, T, M, V, W, ws, nrm, cfg):
    """Runs one entry point on the guarded views; returns the extra guarded
    buffers it used."""
    d = _dpz()
    P = N * C
    g, t, m, v, w, s, o = G.view, T.view, M.view, V.view, W.view, ws.view, nrm.view
    if name == "reduce_scatter":
        d.dp_reduce_scatter_avg(g, N)
    elif name == "allreduce":
        d.dp_allreduce_avg(g, N)
    elif name == "norm":
        d.dp_reduce_scatter_avg(g, N)
        d.dp_grad_global_norm(g, N, s, o)
    elif name == "norm_static":
        d.dp_reduce_scatter_avg(g, N)
        d.dp_grad_global_norm_static(g, N, o)
    elif name == "adamw_owner":
        d.dp_reduce_scatter_avg(g, N)
        d.dp_grad_global_norm(g, N, s, o)
        d.zero1_adamw_step(g, t, m, v, w, N, cfg, ws=s)
    elif name == "allgather":
        d.dp_allgather(w, N)
    elif name == "step_clip":
        d.dp_zero1_step(g, t, m, v, w, N, cfg, ws=s, norm_out=o)
    elif name == "step_no_clip":
        d.dp_zero1_step(g, t, m, v, w, N, _no_clip(cfg), ws=s, norm_out=o)
    elif name == "step_no_clip_no_ws":
        d.dp_zero1_step(g, t, m, v, w, N, _no_clip(cfg))
    elif name == "buckets":
        half = (C // 2 // 256) * 256
        for c in range(N):           # two ranges per chunk, each on segment boundaries
            d.dp_reduce_scatter_avg_range(g, N, c * C, half, ws=s)
            d.dp_reduce_scatter_avg_range(g, N, c * C + half, C - half, ws=s)
        d.dp_grad_norm_finalize(s, P, N, o)
        d.dp_zero1_update(g, t, m, v, w, N, cfg, ws=s)
    elif name == "zero2":
        shards = Guarded(P, g.dtype)
        d.dp_reduce_scatter_avg_bucket(g, 0, shards.view, N, ws=s)
        d.dp_grad_norm_finalize(s, P, N, o)
        d.dp_zero2_update(shards.view, t, m, v, w, N, cfg, ws=s)
        return [shards]
    else:
        raise ValueError(name)
    return []


ENTRIES = ["reduce_scatter", "allreduce", "norm", "norm_static", "adamw_owner", "allgather",
           "step_clip", "step_no_clip", "step_no_clip_no_ws", "buckets", "zero2"]


@pytest.mark.parametrize("C", [2056, 1032])
@pytest.mark.parametrize("gdt,wdt", [("bf16", "bf16"), ("f32", "f32")])
@pytest.mark.parametrize("name", ENTRIES)
def test_every_entry_point_keeps_its_guard_bands(name, gdt, wdt, C):
    bufs = _problem(C, gdt, wdt)
    extra = _entry(name, C, *bufs)
    torch.cuda.synchronize()
    names = ["grads", "master", "m", "v", "weights", "ws", "norm_out"]
    for nm, b in list(zip(names, bufs[:7])) + [("shards", x) for x in extra]:
        assert b.intact(), f"{name}: a byte next to {nm} changed"
    if name not in ("reduce_scatter", "allreduce", "allgather", "norm_static",
                    "step_no_clip_no_ws"):
        assert _dpz().ws_status(bufs[5].view) == 0
    assert _dpz().device_status() == 0
    nrm = bufs[6].view.item()
    if name in ("reduce_scatter", "allreduce", "allgather", "step_no_clip_no_ws"):
        assert bufs[6].view.view(torch.uint8).tolist() == [0xA5] * 4    # norm_out not written
    else:
        assert np.isfinite(nrm) and nrm > 0.0
