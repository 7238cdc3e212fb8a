"""Buckets and ZeRO-2 on the GPU.

A simulated backward pass writes the gradients bucket by bucket, last
layer first, on the main stream and records an event after each bucket; a
second stream waits on each event and reduces that bucket while the next one
is being written ("A4 — Multi-GPU with NCCL and ZeRO-1", Part 3; "Lab 09 —
Parallelism, simulated", §2).  ZeRO-2 reduces each bucket from a staging
buffer, reused for every bucket, into compact gradient shards.  Both must
give, bit for bit, what the whole-arena dp_zero1_step gives."""
import numpy as np
import pytest
import torch

import inputs as I
import oracle as O

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import gradient_reduction_zero_gb300.dpz as dpz
    from gpu_util import DEV, check_step, down, same_bits, up


def segment_buckets(P, N, nb, seed):
    """nb buckets covering [0, P) whose bounds sit on 256-element segment
    boundaries of their chunks, in backward (reverse) order."""
    C = P // N
    bounds = sorted({c * C + k for c in range(N) for k in range(0, C, 256)} | {P})
    rng = np.random.default_rng(seed)
    inner = sorted(rng.choice(bounds[1:-1], size=min(nb - 1, len(bounds) - 2), replace=False))
    edges = [0] + [int(b) for b in inner] + [P]
    return [(edges[i], edges[i + 1] - edges[i]) for i in range(len(edges) - 1)][::-1]


def problem(N, C, clip, seed):
    w = I.TINY.with_(N=N, P=N * C, gdtype="bf16", wdtype="bf16",
                     grad=I.Dist(I.NORMAL_TAIL, 1e-3), grad_seed=seed,
                     m=I.Dist(I.NORMAL, 1e-4), v=I.Dist(I.ABS_NORMAL, 1e-6), lr=1.5e-4,
                     beta1=0.9, beta2=0.95, step=1000, clip=clip)
    g = I.arena_host(w)
    th, m, v = (I.state_host(w, k) for k in ("master", "m", "v"))
    return w, g, th, m, v


def fused_reference(w, g, th, m, v, acc32):
    G, T, M, V = up(g), up(th), up(m), up(v)
    W = torch.zeros(w.N * w.P, dtype=torch.bfloat16, device=DEV)
    ws = dpz.workspace(w.P, w.N, DEV)
    nrm = torch.zeros(1, device=DEV)
    cfg = dpz.make_cfg(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.step, w.clip,
                       store_avg=True)
    dpz.dp_zero1_step(G, T, M, V, W, w.N, cfg, ws=ws, norm_out=nrm, acc32=acc32)
    torch.cuda.synchronize()
    return down(G), down(T), down(M), down(V), down(W), nrm.item()


@pytest.mark.parametrize("N,C,nb", [(4, 6152, 7), (8, 2056, 5), (3, 1000, 4), (7, 1032, 6),
                                    (4, 262_144, 12)])
@pytest.mark.parametrize("clip", [0.0, 1e-3])
@pytest.mark.parametrize("acc32", [False, True])
@pytest.mark.parametrize("max_ctas", [0, 1, 152])
def test_bucketed_zero1_matches_whole_arena(N, C, nb, clip, acc32, max_ctas):
    """max_ctas = 1: one block per chunk piece loops over the whole piece;
    152: one block per SM; 0: one pass."""
    w, g, th, m, v = problem(N, C, clip, seed=N + nb)
    ref = fused_reference(w, g, th, m, v, acc32)
    P = w.P
    src = up(g).view(N, P)                      # what backward will produce
    G = torch.zeros(N, P, dtype=torch.bfloat16, device=DEV)
    T, M, V = up(th), up(m), up(v)
    W = torch.zeros(N * P, dtype=torch.bfloat16, device=DEV)
    ws = dpz.workspace(P, N, DEV)
    nrm = torch.zeros(1, device=DEV)
    cfg = dpz.make_cfg(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.step, w.clip)
    main = torch.cuda.current_stream()
    comm = torch.cuda.Stream()
    for lo, n in segment_buckets(P, N, nb, seed=nb):
        G[:, lo:lo + n].copy_(src[:, lo:lo + n])           # "backward" writes the bucket
        ev = torch.cuda.Event()
        ev.record(main)
        comm.wait_event(ev)                                 # never reduce before it exists
        dpz.dp_reduce_scatter_avg_range(G, N, lo, n, ws=ws, stream=comm, acc32=acc32,
                                        max_ctas=max_ctas)
    dpz.dp_grad_norm_finalize(ws, P, N, nrm, stream=comm)
    dpz.dp_zero1_update(G, T, M, V, W, N, cfg, ws=ws, stream=comm)
    main.wait_stream(comm)
    torch.cuda.synchronize()
    Gd = down(G)
    for c in range(N):
        sl = slice(c * C, (c + 1) * C)
        assert same_bits(Gd[c, sl], ref[0][c, sl])
    out = (Gd.reshape(N, P), down(T), down(M), down(V), down(W).reshape(N, P), nrm.item())
    for got, want in zip(out[1:5], ref[1:5]):
        assert same_bits(got.reshape(want.shape), want)
    assert nrm.item() == ref[5]
    assert dpz.ws_status(ws) == 0
    # and directly against the oracle's step on the same inputs
    check_step(w, g, th, m, v, np.zeros((N, P), dtype=np.uint16), out, acc32=acc32)


@pytest.mark.parametrize("N,C,nb", [(4, 6152, 7), (8, 2056, 5), (3, 1000, 4), (4, 262_144, 12)])
@pytest.mark.parametrize("clip", [0.0, 1e-3])
@pytest.mark.parametrize("acc32", [False, True])
@pytest.mark.parametrize("max_ctas", [0, 2])
def test_zero2_matches_zero1(N, C, nb, clip, acc32, max_ctas):
    w, g, th, m, v = problem(N, C, clip, seed=2 * N + nb)
    ref = fused_reference(w, g, th, m, v, acc32)
    P = w.P
    src = up(g).view(N, P)
    buckets = segment_buckets(P, N, nb, seed=3 * nb)
    cap = max(n for _, n in buckets)
    staging = torch.zeros(N * cap, dtype=torch.bfloat16, device=DEV)   # reused per bucket
    shards = torch.zeros(P, dtype=torch.bfloat16, device=DEV)
    T, M, V = up(th), up(m), up(v)
    W = torch.zeros(N * P, dtype=torch.bfloat16, device=DEV)
    ws = dpz.workspace(P, N, DEV)
    nrm = torch.zeros(1, device=DEV)
    cfg = dpz.make_cfg(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.step, w.clip)
    main = torch.cuda.current_stream()
    comm = torch.cuda.Stream()
    done = None
    for lo, n in buckets:
        if done is not None:
            main.wait_event(done)               # the previous bucket has left the staging buffer
        stage = staging[:N * n]
        stage.view(N, n).copy_(src[:, lo:lo + n])
        ready = torch.cuda.Event()
        ready.record(main)
        comm.wait_event(ready)
        dpz.dp_reduce_scatter_avg_bucket(stage, lo, shards, N, ws=ws, stream=comm, acc32=acc32,
                                         max_ctas=max_ctas)
        done = torch.cuda.Event()
        done.record(comm)
    dpz.dp_grad_norm_finalize(ws, P, N, nrm, stream=comm)
    dpz.dp_zero2_update(shards, T, M, V, W, N, cfg, ws=ws, stream=comm)
    main.wait_stream(comm)
    torch.cuda.synchronize()
    owner_avg = np.concatenate([ref[0][c, c * C:(c + 1) * C] for c in range(N)])
    assert same_bits(down(shards), owner_avg)
    out = (None, down(T), down(M), down(V), down(W).reshape(N, P), nrm.item())
    for got, want in zip(out[1:5], ref[1:5]):
        assert same_bits(got.reshape(want.shape), want)
    assert nrm.item() == ref[5]
    assert dpz.ws_status(ws) == 0
    # the shards are the oracle's reduce-scatter, and the update its ZeRO-1 step
    a = g.copy()
    O.reduce_scatter_avg(a, acc32=acc32)
    assert same_bits(down(shards), np.concatenate([a[c, c * C:(c + 1) * C] for c in range(N)]))
    check_step(w, g, th, m, v, np.zeros((N, P), dtype=np.uint16), out, check_avg=False,
               acc32=acc32)


def test_range_without_partials_any_alignment():
    """Without ws the ranges only need 8-element alignment."""
    N, C = 4, 1000
    w, g, th, m, v = problem(N, C, 0.0, seed=11)
    P = w.P
    G = up(g)
    for lo, n in [(0, 1000), (1000, 1008), (2008, 992), (3000, 1000)]:
        dpz.dp_reduce_scatter_avg_range(G, N, lo, n)
    torch.cuda.synchronize()
    a = g.copy()
    O.reduce_scatter_avg(a)
    out = down(G).reshape(N, P)
    for c in range(N):
        sl = slice(c * C, (c + 1) * C)
        assert same_bits(out[c, sl], a[c, sl])


@pytest.mark.parametrize("N,C,gdt,acc32", [(1, 4104, "bf16", False), (1, 4104, "bf16", True),
                                           (2, 2056, "bf16", False), (2, 2056, "bf16", True),
                                           (7, 1032, "bf16", False), (7, 1032, "bf16", True),
                                           (8, 776, "bf16", True), (12, 520, "bf16", False),
                                           (5, 2000, "f32", False), (8, 776, "f32", False),
                                           (12, 520, "f32", False), (16, 264, "f32", False)])
def test_range_partials_match_whole_arena(N, C, gdt, acc32):
    """Every register bound of the range kernel (compile-time N up to 8, the
    run-time fold beyond, both storage dtypes, fp32 accumulation): the ranges'
    averages are the oracle's, bit for bit, and the norm from their partials
    equals the norm of the whole-arena reduce.  At N = 1 and 2 with bf16
    storage the whole-arena reduce takes two segments per warp; 17 and 18
    segments leave the last warp half idle and make warps straddle chunks."""
    w = I.TINY.with_(N=N, P=N * C, gdtype=gdt, grad=I.Dist(I.NORMAL, 1e-3), grad_seed=N + C)
    g = I.arena_host(w)
    P = w.P
    G = up(g)
    ws = dpz.workspace(P, N, DEV)
    for lo, n in segment_buckets(P, N, 5, seed=N):
        dpz.dp_reduce_scatter_avg_range(G, N, lo, n, ws=ws, acc32=acc32)
    nrm = torch.zeros(1, device=DEV)
    dpz.dp_grad_norm_finalize(ws, P, N, nrm)
    G2 = up(g)
    ws2 = dpz.workspace(P, N, DEV)
    nrm2 = torch.zeros(1, device=DEV)
    dpz.dp_reduce_scatter_avg(G2, N, acc32=acc32)
    dpz.dp_grad_global_norm(G2, N, ws2, nrm2)
    torch.cuda.synchronize()
    a = g.copy()
    O.reduce_scatter_avg(a, acc32=acc32)
    out, out2 = down(G).reshape(N, P), down(G2).reshape(N, P)
    for c in range(N):
        sl = slice(c * C, (c + 1) * C)
        assert same_bits(out[c, sl], a[c, sl])
        assert same_bits(out2[c, sl], a[c, sl])
    assert nrm.item() == nrm2.item() and nrm.item() > 0
