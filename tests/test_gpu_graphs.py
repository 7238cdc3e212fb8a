"""The step captured in a CUDA graph and replayed: the calls only enqueue
kernels on the caller's stream (no allocation, no host synchronisation), so
a captured step replays with the same bits as eager calls, and its first
replay is the oracle's step.  The tiny workload is launch-latency bound,
which is where replaying a graph pays ("Distributed training", "Overlap and
graphs": one CUDA graph per GPU)."""
import numpy as np
import pytest
import torch

import inputs as I
import oracle as O

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import gradient_reduction_zero_gb300.dpz as dpz
    from gpu_util import DEV, check_step, down, same_bits, up


def _inputs(w):
    g = I.arena_host(w)
    th, m, v = (I.state_host(w, k) for k in ("master", "m", "v"))
    wts = np.zeros((w.N, w.P), dtype=np.uint16 if w.wdtype == "bf16" else np.float32)
    return g, th, m, v, wts


@pytest.mark.parametrize("clip,acc32", [(0.0, False), (1e-3, False), (1e-3, True)])
@pytest.mark.parametrize("N,C", [(4, 1024), (8, 2056), (3, 1000)])
def test_zero1_step_graph_replay_matches_eager(N, C, clip, acc32):
    w = I.TINY.with_(N=N, P=N * C, gdtype="bf16", wdtype="bf16", grad=I.Dist(I.NORMAL_TAIL, 1e-3),
                     m=I.Dist(I.NORMAL, 1e-4), v=I.Dist(I.ABS_NORMAL, 1e-6), step=7, clip=clip)
    cfg = dpz.make_cfg(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.step, w.clip)
    host = _inputs(w)
    eager = [up(x) for x in host]
    graph = [t.clone() for t in eager]
    ws_e, ws_g = dpz.workspace(w.P, N, DEV), dpz.workspace(w.P, N, DEV)
    n_e = torch.zeros(1, device=DEV)
    n_g = torch.zeros(1, device=DEV)
    reps = 3
    for _ in range(reps):
        dpz.dp_zero1_step(*eager, N, cfg, ws=ws_e, norm_out=n_e, acc32=acc32)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        dpz.dp_zero1_step(*graph, N, cfg, ws=ws_g, norm_out=n_g, acc32=acc32)
    # capture records the kernels without running them: the first replay is
    # the first step, the oracle's step on the same inputs
    g.replay()
    torch.cuda.synchronize()
    first = [down(t) for t in graph] + [n_g.item()]
    first[0] = first[0].reshape(N, w.P)
    first[4] = first[4].reshape(N, w.P)
    check_step(w, *host, tuple(first), check_avg=clip > 0, acc32=acc32)
    if clip <= 0:
        assert same_bits(first[0], host[0])       # no averages stored without clip
    assert dpz.ws_status(ws_g) == 0
    for _ in range(reps - 1):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, graph):
        assert same_bits(down(a), down(b))
    assert n_e.item() == n_g.item()


def test_allreduce_graph_replay_matches_eager():
    w = I.allreduce_sweep(64 * 1024, 8)
    g0 = I.arena_host(w)
    A = up(g0)
    B = up(g0)
    dpz.dp_allreduce_avg(A, w.N)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        dpz.dp_allreduce_avg(B, w.N)
    graph.replay()
    torch.cuda.synchronize()
    assert same_bits(down(A), down(B))
    ref = g0.copy()
    O.ring_allreduce_avg(ref)
    assert same_bits(down(B), ref)
