"""GPU parity at the workloads' full sizes, in the launch configurations the
benchmark times (dp_zero1_step with clip, workspace and norm output; also
without clip, the one-kernel step, and with the fp32-accumulating ring;
dp_allreduce_avg for the all-reduce workloads).  The oracle computes sampled
windows of every chunk one by one (the start, the middle and the ragged end)
and the global norm over the whole arena, window by window on host threads;
the rest is checked through properties that hold at any size (non-owner
chunks untouched, every weight replica identical)."""
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import inputs as I
import oracle as O

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

if torch.cuda.is_available():
    import gradient_reduction_zero_gb300.dpz as dpz
    from gpu_util import (DEV, assert_close_tol, assert_weights, down, f32_view, same_bits,
                          state_tolerances)

WIDTH = 4096


def window_offsets(C):
    return sorted({0, (C // 2) // 8 * 8, C - WIDTH})


def oracle_full_sumsq(w, width=1 << 20, acc32=False):
    """Sum of squares of the averaged gradient of the whole arena: the oracle's
    reduce-scatter, average and sum of squares on every window, added with
    math.fsum (the sum of squares is additive over windows)."""
    C = w.C

    def part(o):
        wd = min(width, C - o)
        g = I.window_arena_host(w, o, wd)
        O.reduce_scatter_avg(g, acc32=acc32)
        return O.sumsq_owned(g)

    with ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        parts = list(ex.map(part, range(0, C, width)))
    return math.fsum(parts)


def gpu_window(t, N, P, C, o, wd):
    """[N][N*wd] of a device arena [N*P]: window [c*C+o, +wd) of every chunk."""
    v = t.view(N, P)
    return np.concatenate([down(v[:, c * C + o:c * C + o + wd]) for c in range(N)], axis=1)


def gpu_state_window(t, N, C, o, wd):
    return np.concatenate([down(t[c * C + o:c * C + o + wd]) for c in range(N)])


@pytest.mark.parametrize("w,acc32", [(I.GPT2_124M, False), (I.GPT2_1P5B, False),
                                     (I.GPT2_1P5B.with_(clip=0.0), False),
                                     (I.GPT2_124M, True)],
                         ids=["gpt2-124m", "gpt2-1.5b", "gpt2-1.5b-no-clip", "gpt2-124m-acc32"])
def test_zero1_step_full_size(w, acc32):
    """The clipped three-kernel step, the one-kernel step without clipping,
    and the fp32-accumulating ring, at full size."""
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

    ss = oracle_full_sumsq(w, acc32=acc32)
    onorm, oscale = O.clip_scale(ss, w.clip)
    assert abs(gnorm - onorm) <= 1e-6 * onorm, (gnorm, onorm)
    if w.clip > 0:
        assert oscale < 1.0                       # the clip is active

    ocfg = O.cfg_from_workload(w)
    for o in window_offsets(C):
        g = I.window_arena_host(w, o, WIDTH)
        th = I.window_state_host(w, "master", o, WIDTH)
        m = I.window_state_host(w, "m", o, WIDTH)
        v = I.window_state_host(w, "v", o, WIDTH)
        wt = np.zeros((N, N * WIDTH), dtype=np.uint16)
        G1, T1, M1, V1, W1 = g.copy(), th.copy(), m.copy(), v.copy(), wt.copy()
        n1, s1, _, _ = O.zero1_step(G1, T1, M1, V1, W1, ocfg, ext_sumsq=ss, acc32=acc32)
        assert n1 == onorm
        Gg = gpu_window(G, N, P, C, o, WIDTH)
        Wg = gpu_window(W, N, P, C, o, WIDTH)
        Tg = gpu_state_window(T, N, C, o, WIDTH)
        Mg = gpu_state_window(M, N, C, o, WIDTH)
        Vg = gpu_state_window(V, N, C, o, WIDTH)
        for c in range(N):
            sl = slice(c * WIDTH, (c + 1) * WIDTH)
            for r in range(N):
                want = G1[c, sl] if r == c else g[r, sl]    # owner: average; others: untouched
                assert same_bits(Gg[r, sl], want), (o, r, c)
        for r in range(N):
            assert same_bits(Wg[r], Wg[0])
        if gnorm == onorm or w.clip <= 0:
            assert same_bits(Tg, T1) and same_bits(Mg, M1) and same_bits(Vg, V1)
            assert same_bits(Wg, W1)
        else:
            avg = np.concatenate([f32_view(G1[c, c * WIDTH:(c + 1) * WIDTH]) for c in range(N)])
            tm, tv, tt = state_tolerances(avg, oscale, th, m, v, M1, V1, ocfg)
            assert_close_tol(Mg, M1, tm, "m")
            assert_close_tol(Vg, V1, tv, "v")
            assert_close_tol(Tg, T1, tt, "master")
            assert_weights(Wg, W1, exact=False)
    del G, T, M, V, W
    torch.cuda.empty_cache()


def _allreduce_full(w):
    N, P, C = w.N, w.P, w.C
    G = torch.empty(N * P, dtype=torch.bfloat16 if w.gdtype == "bf16" else torch.float32,
                    device=DEV)
    I.fill_grads_device(w, G)
    dpz.dp_allreduce_avg(G, N)
    torch.cuda.synchronize()
    wd = min(WIDTH, C)
    for o in sorted({0, (C // 2) // 8 * 8, C - wd}):
        g = I.window_arena_host(w, o, wd)
        O.ring_allreduce_avg(g)
        assert same_bits(gpu_window(G, N, P, C, o, wd), g), o
    del G
    torch.cuda.empty_cache()


def test_allreduce_7b_full_size():
    _allreduce_full(I.ALLREDUCE_7B)


@pytest.mark.parametrize("N", [2, 4, 8])
def test_allreduce_sweep(N):
    for size in I.SWEEP_SIZES:
        w = I.allreduce_sweep(size, N)
        if w.P <= 1 << 20:
            # small enough for the whole arena
            g = I.arena_host(w)
            G = torch.from_numpy(g.reshape(-1).copy()).to(DEV)
            dpz.dp_allreduce_avg(G, N)
            O.ring_allreduce_avg(g)
            assert same_bits(down(G).reshape(N, w.P), g), size
        else:
            _allreduce_full(w)
