"""GPU parity at the workloads' full sizes, on every element, in the launch
configurations the benchmark times (dp_zero1_step with clip, workspace and
norm output; also without clip, the one-kernel step, and with the
fp32-accumulating ring; dp_allreduce_avg for the all-reduce workloads).

The oracle runs window by window (oracle_windows): the windows tile every
chunk, so every averaged gradient, every untouched non-owner element, every
master/m/v value and every weight of every replica is compared.  Host threads
run the oracle on the windows while the matching device windows are copied
down, so host memory stays bounded (a few hundred MB per thread)."""
import math

import numpy as np
import pytest
import torch

import inputs as I
import oracle as O
from oracle_windows import for_every_window, oracle_full_sumsq, remember_sumsq

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

if torch.cuda.is_available():
    import gradient_reduction_zero_gb300.dpz as dpz
    from gpu_util import (DEV, assert_close_tol, assert_weights, down, f32_view, same_bits,
                          state_tolerances)


def first_difference(got, want):
    """Index and values of the first element whose bits differ (NaN matches
    NaN)."""
    fa, fb = f32_view(got).ravel(), f32_view(want).ravel()
    ia = got.ravel().view(np.uint16 if got.dtype == np.uint16 else np.uint32)
    ib = want.ravel().view(np.uint16 if want.dtype == np.uint16 else np.uint32)
    bad = (ia != ib) & ~(np.isnan(fa) & np.isnan(fb))
    i = int(np.argmax(bad))
    return i, fa[i], fb[i]


def assert_same(got, want, what):
    if not same_bits(got, want):
        i, a, b = first_difference(got, want)
        raise AssertionError(f"{what}: element {i} of the window differs (gpu {a}, oracle {b})")


def gpu_window(t, N, P, C, o, wd):
    """[N][N*wd] of a device arena [N*P]: window [c*C+o, +wd) of every chunk."""
    v = t.view(N, P)
    return np.concatenate([down(v[:, c * C + o:c * C + o + wd]) for c in range(N)], axis=1)


def gpu_state_window(t, N, C, o, wd):
    return np.concatenate([down(t[c * C + o:c * C + o + wd]) for c in range(N)])


@pytest.mark.parametrize("w,acc32", [(I.GPT2_124M, False),
                                     (I.GPT2_1P5B.with_(clip=0.0), False),
                                     (I.GPT2_1P5B, False),
                                     (I.GPT2_124M, True)],
                         ids=["gpt2-124m", "gpt2-1.5b-no-clip", "gpt2-1.5b", "gpt2-124m-acc32"])
def test_zero1_step_full_size(w, acc32):
    """The clipped three-kernel step, the one-kernel step without clipping,
    and the fp32-accumulating ring, at full size, every element against the
    oracle."""
    N, P, C = w.N, w.P, w.C
    gd = torch.bfloat16
    G = torch.empty(N * P, dtype=gd, device=DEV)
    I.fill_grads_device(w, G)
    T = torch.empty(P, dtype=torch.float32, device=DEV)
    M, V = torch.empty_like(T), torch.empty_like(T)
    for which, t in (("master", T), ("m", M), ("v", V)):
        I.fill_state_device(w, which, t)
    W = torch.zeros(N * P, dtype=gd, device=DEV)
    ws = dpz.workspace(P, N, DEV)
    nrm = torch.zeros(1, device=DEV)
    cfg = dpz.make_cfg(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.step, w.clip,
                       store_avg=True)
    dpz.dp_zero1_step(G, T, M, V, W, N, cfg, ws=ws, norm_out=nrm, acc32=acc32)
    torch.cuda.synchronize()
    gnorm = nrm.item()
    assert dpz.ws_status(ws) == 0
    # the standalone norm (bulk-copy staged kernel) of the stored averages is
    # the same float: the same per-segment partials, summed in the same order
    ws2, nrm2 = dpz.workspace(P, N, DEV), torch.zeros(1, device=DEV)
    dpz.dp_grad_global_norm(G, N, ws2, nrm2)
    torch.cuda.synchronize()
    assert nrm2.item() == gnorm
    assert dpz.ws_status(ws2) == 0
    assert dpz.device_status() == 0
    del ws2

    # without clipping the update does not depend on the norm, so the windows
    # run in one pass that also yields the sum of squares; with clipping the
    # oracle needs the whole arena's sum of squares first
    ss = oracle_full_sumsq(w, acc32) if w.clip > 0 else None
    onorm, oscale = O.clip_scale(ss, w.clip) if ss is not None else (None, 1.0)
    exact = w.clip <= 0 or gnorm == onorm
    ocfg = O.cfg_from_workload(w)

    def check(o, wd):
        g = I.window_arena_host(w, o, wd)
        th = I.window_state_host(w, "master", o, wd)
        m = I.window_state_host(w, "m", o, wd)
        v = I.window_state_host(w, "v", o, wd)
        wt = np.zeros((N, N * wd), dtype=np.uint16)
        G1, T1, M1, V1, W1 = g.copy(), th.copy(), m.copy(), v.copy(), wt
        O.zero1_step(G1, T1, M1, V1, W1, ocfg, ext_sumsq=-1.0 if ss is None else ss,
                     acc32=acc32)
        Gg = gpu_window(G, N, P, C, o, wd)
        Wg = gpu_window(W, N, P, C, o, wd)
        Tg = gpu_state_window(T, N, C, o, wd)
        Mg = gpu_state_window(M, N, C, o, wd)
        Vg = gpu_state_window(V, N, C, o, wd)
        for c in range(N):
            sl = slice(c * wd, (c + 1) * wd)
            for r in range(N):
                want = G1[c, sl] if r == c else g[r, sl]   # owner: average; others: untouched
                assert_same(Gg[r, sl], want, f"grads slab {r} chunk {c} window {o}")
        if exact:
            assert_same(Tg, T1, f"master window {o}")
            assert_same(Mg, M1, f"m window {o}")
            assert_same(Vg, V1, f"v window {o}")
            for r in range(N):
                assert_same(Wg[r], W1[r], f"weights slab {r} window {o}")
        else:
            avg = np.concatenate([f32_view(G1[c, c * wd:(c + 1) * wd]) for c in range(N)])
            tm, tv, tt = state_tolerances(avg, oscale, th, m, v, M1, V1, ocfg)
            assert_close_tol(Mg, M1, tm, "m")
            assert_close_tol(Vg, V1, tv, "v")
            assert_close_tol(Tg, T1, tt, "master")
            assert_weights(Wg, W1, exact=False)
        return O.sumsq_owned(G1)          # this window's part of the sum of squares

    parts = for_every_window(C, check)
    total = math.fsum(parts)
    if ss is None:
        remember_sumsq(w, acc32, total)
        onorm, _ = O.clip_scale(total, 0.0)
    else:
        assert total == ss
        assert oscale < 1.0                       # the clip is active
    assert abs(gnorm - onorm) <= 1e-6 * onorm, (gnorm, onorm)
    del G, T, M, V, W
    torch.cuda.empty_cache()


def _allreduce_full(w):
    """dp_allreduce_avg on the whole arena; every element of every slab
    against the oracle's ring all-reduce, window by window."""
    N, P, C = w.N, w.P, w.C
    G = torch.empty(N * P, dtype=torch.bfloat16 if w.gdtype == "bf16" else torch.float32,
                    device=DEV)
    I.fill_grads_device(w, G)
    dpz.dp_allreduce_avg(G, N)
    torch.cuda.synchronize()

    def check(o, wd):
        g = I.window_arena_host(w, o, wd)
        O.ring_allreduce_avg(g)
        assert_same(gpu_window(G, N, P, C, o, wd), g, f"all-reduce window {o}")

    for_every_window(C, check)
    del G
    torch.cuda.empty_cache()


def test_allreduce_7b_full_size():
    _allreduce_full(I.ALLREDUCE_7B)


@pytest.mark.parametrize("N", [2, 4, 8])
def test_allreduce_sweep(N):
    for size in I.SWEEP_SIZES:
        w = I.allreduce_sweep(size, N)
        if w.P <= 1 << 20:
            # small enough for the whole arena at once
            g = I.arena_host(w)
            G = torch.from_numpy(g.reshape(-1).copy()).to(DEV)
            dpz.dp_allreduce_avg(G, N)
            O.ring_allreduce_avg(g)
            assert same_bits(down(G).reshape(N, w.P), g), size
        else:
            _allreduce_full(w)


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def _segment_buckets(P, N, k):
    """k buckets on 256-element segment boundaries of their chunks, in
    backward (last-first) order."""
    C = P // N
    edges = {0, P}
    for i in range(1, k):
        b = P * i // k
        c = b // C
        edges.add(c * C + (b - c * C) // 256 * 256)
    edges = sorted(edges)
    return [(edges[i], edges[i + 1] - edges[i]) for i in range(len(edges) - 1)][::-1]


def test_buckets_and_zero2_full_size():
    """The GPT-2 1.5B step in 16 buckets reduced on a side stream with the grid
    capped at one block per SM (the bench's overlap configuration), then the
    norm and dp_zero1_update; and as ZeRO-2 from a reused staging buffer into
    gradient shards.  Both equal dp_zero1_step bit for bit on every element:
    the same partials, the same norm, the same averages, master/m/v and
    weights.  (dp_zero1_step itself is compared with the oracle on every
    element above.)"""
    w = I.GPT2_1P5B
    N, P, C = w.N, w.P, w.C
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    cfg = dpz.make_cfg(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.step, w.clip,
                       store_avg=True)

    def fresh():
        G = torch.empty(N * P, dtype=torch.bfloat16, device=DEV)
        I.fill_grads_device(w, G)
        T = torch.empty(P, dtype=torch.float32, device=DEV)
        M, V = torch.empty_like(T), torch.empty_like(T)
        for which, t in (("master", T), ("m", M), ("v", V)):
            I.fill_state_device(w, which, t)
        return G, T, M, V, torch.zeros(N * P, dtype=torch.bfloat16, device=DEV)

    G, T, M, V, W = fresh()
    ws = dpz.workspace(P, N, DEV)
    nrm = torch.zeros(1, device=DEV)
    dpz.dp_zero1_step(G, T, M, V, W, N, cfg, ws=ws, norm_out=nrm)
    owner = torch.cat([G.view(N, P)[c, c * C:(c + 1) * C] for c in range(N)])
    del G
    torch.cuda.empty_cache()

    buckets = _segment_buckets(P, N, 16)
    main = torch.cuda.current_stream()
    comm = torch.cuda.Stream()

    # ZeRO-1 in buckets, in place in the arena
    Gb, Tb, Mb, Vb, Wb = fresh()
    wsb = dpz.workspace(P, N, DEV)
    nrmb = torch.zeros(1, device=DEV)
    comm.wait_stream(main)
    for lo, n in buckets:
        dpz.dp_reduce_scatter_avg_range(Gb, N, lo, n, ws=wsb, stream=comm, max_ctas=sms)
    dpz.dp_grad_norm_finalize(wsb, P, N, nrmb, stream=comm)
    dpz.dp_zero1_update(Gb, Tb, Mb, Vb, Wb, N, cfg, ws=wsb, stream=comm)
    main.wait_stream(comm)
    torch.cuda.synchronize()
    assert nrmb.item() == nrm.item()
    assert dpz.ws_status(wsb) == 0
    owner_b = torch.cat([Gb.view(N, P)[c, c * C:(c + 1) * C] for c in range(N)])
    assert torch.equal(_bits(owner_b), _bits(owner))
    for got, want in ((Tb, T), (Mb, M), (Vb, V), (Wb, W)):
        assert torch.equal(_bits(got), _bits(want))
    del owner_b, Gb, Tb, Mb, Vb, Wb
    torch.cuda.empty_cache()

    # ZeRO-2: each bucket's N rows staged in one reused buffer, reduced into shards
    src, T2, M2, V2, W2 = fresh()
    src = src.view(N, P)
    ws2 = dpz.workspace(P, N, DEV)
    nrm2 = torch.zeros(1, device=DEV)
    shards = torch.zeros(P, dtype=torch.bfloat16, device=DEV)
    staging = torch.empty(N * max(n for _, n in buckets), dtype=torch.bfloat16, device=DEV)
    for lo, n in buckets:
        stage = staging[:N * n]
        stage.view(N, n).copy_(src[:, lo:lo + n])
        dpz.dp_reduce_scatter_avg_bucket(stage, lo, shards, N, ws=ws2, max_ctas=sms)
    dpz.dp_grad_norm_finalize(ws2, P, N, nrm2)
    dpz.dp_zero2_update(shards, T2, M2, V2, W2, N, cfg, ws=ws2)
    torch.cuda.synchronize()
    assert nrm2.item() == nrm.item()
    assert dpz.ws_status(ws2) == 0
    assert torch.equal(_bits(shards), _bits(owner))
    for got, want in ((T2, T), (M2, M), (V2, V), (W2, W)):
        assert torch.equal(_bits(got), _bits(want))
    assert dpz.device_status() == 0
    del src, T2, M2, V2, W2, shards, staging, T, M, V, W, owner
    torch.cuda.empty_cache()


@pytest.mark.parametrize("clip", [1.0, 0.0], ids=["clip", "no-clip"])
def test_graph_replay_full_size(clip):
    """The GPT-2 1.5B step captured in a CUDA graph (as bench --graph times it)
    and replayed twice equals two eager steps on a fresh copy of the inputs,
    bit for bit on every element: the calls only enqueue kernels, and every
    run of the step is deterministic."""
    w = I.GPT2_1P5B.with_(clip=clip)
    N, P = w.N, w.P
    cfg = dpz.make_cfg(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.step, w.clip)

    def fresh():
        G = torch.empty(N * P, dtype=torch.bfloat16, device=DEV)
        I.fill_grads_device(w, G)
        T = torch.empty(P, dtype=torch.float32, device=DEV)
        M, V = torch.empty_like(T), torch.empty_like(T)
        for which, t in (("master", T), ("m", M), ("v", V)):
            I.fill_state_device(w, which, t)
        return [G, T, M, V, torch.zeros(N * P, dtype=torch.bfloat16, device=DEV)]

    eager = fresh()
    ws_e, n_e = dpz.workspace(P, N, DEV), torch.zeros(1, device=DEV)
    for _ in range(2):
        dpz.dp_zero1_step(*eager, N, cfg, ws=ws_e, norm_out=n_e)
    torch.cuda.synchronize()
    eager_bits = [_bits(t).clone() for t in eager[1:]]     # master, m, v, weights
    del eager
    torch.cuda.empty_cache()

    graph = fresh()
    ws_g, n_g = dpz.workspace(P, N, DEV), torch.zeros(1, device=DEV)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        dpz.dp_zero1_step(*graph, N, cfg, ws=ws_g, norm_out=n_g)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert n_g.item() == n_e.item()
    for got, want in zip(graph[1:], eager_bits):
        assert torch.equal(_bits(got), want)
    assert dpz.device_status() == 0
    del graph, eager_bits, g
    torch.cuda.empty_cache()
