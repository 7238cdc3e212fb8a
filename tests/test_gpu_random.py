"""Seeded random shapes against the oracle: the step (clip or not, the stored
averages or not, bf16 or fp32-accumulating rings, every dtype pair) with both
norm entry points on its averages, and the bucketed path on random splits of
the arena into segment-aligned ranges reduced in random order.

Each case draws N from 1..64, a chunk of 8 to 262,144 elements (mostly small,
so that the oracle stays fast), the dtypes and the modes from one seed; the
case's id names the seed, so a failure can be re-run alone."""
import numpy as np
import pytest
import torch

import inputs as I
from gpu_util import DEV, check_step, down, up

pytestmark = pytest.mark.gpu

NS = [1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 16, 24, 32, 48, 64]
DTYPES = [("bf16", "bf16"), ("f32", "bf16"), ("f32", "f32"), ("bf16", "f32")]


def _dpz():
    import gradient_reduction_zero_gb300.dpz as dpz
    return dpz


def _case(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.choice(NS))
    big = rng.random() < 0.15
    C = 8 * int(rng.integers(4000, 32768)) if big and N <= 8 else 8 * int(rng.integers(1, 4000))
    gdt, wdt = DTYPES[int(rng.integers(0, 4))]
    clip = float(rng.choice([0.0, 1e-3, 1e3]))
    acc32 = gdt == "bf16" and bool(rng.integers(0, 2))
    store_avg = bool(rng.integers(0, 2))
    w = I.TINY.with_(N=N, P=N * C, gdtype=gdt, wdtype=wdt, clip=clip,
                     grad=I.Dist(I.NORMAL_TAIL, 1e-3), grad_seed=int(rng.integers(0, 1 << 30)),
                     m=I.Dist(I.NORMAL, 1e-4), v=I.Dist(I.ABS_NORMAL, 1e-6), lr=1.5e-4,
                     beta1=0.9, beta2=0.95, step=int(rng.integers(1, 2000)))
    return w, acc32, store_avg, rng


def _inputs(w):
    g = I.arena_host(w)
    th, m, v = (I.state_host(w, k) for k in ("master", "m", "v"))
    wts = np.zeros((w.N, w.P), dtype=np.uint16 if w.wdtype == "bf16" else np.float32)
    return g, th, m, v, wts


@pytest.mark.parametrize("seed", [1000 + k for k in range(100)])
def test_random_step_matches_oracle(seed):
    dpz = _dpz()
    w, acc32, store_avg, _ = _case(seed)
    N = w.N
    g, th, m, v, wts = _inputs(w)
    G, T, M, V, W = up(g), up(th), up(m), up(v), up(wts)
    ws = dpz.workspace(w.P, N, DEV)
    nrm = torch.full((1,), -1.0, device=DEV)
    cfg = dpz.make_cfg(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.step, w.clip,
                       store_avg=store_avg)
    dpz.dp_zero1_step(G, T, M, V, W, N, cfg, ws=ws, norm_out=nrm, acc32=acc32)
    torch.cuda.synchronize()
    assert dpz.ws_status(ws) == 0
    out = (down(G).reshape(N, w.P), down(T), down(M), down(V), down(W).reshape(N, w.P),
           nrm.item())
    check_step(w, g, th, m, v, wts, out, check_avg=store_avg or w.clip > 0, acc32=acc32)
    if store_avg or w.clip > 0:
        # both norm entry points on the stored averages give the step's norm bits
        ws2 = dpz.workspace(w.P, N, DEV)
        n2 = torch.zeros(1, device=DEV)
        dpz.dp_grad_global_norm(G, N, ws2, n2)
        torch.cuda.synchronize()
        assert n2.item() == out[5], (n2.item(), out[5])
        if dpz.lib.dpz_workspace_bytes(w.P, N) <= 4 << 20:
            n3 = torch.zeros(1, device=DEV)
            dpz.dp_grad_global_norm_static(G, N, n3)
            torch.cuda.synchronize()
            assert n3.item() == out[5], (n3.item(), out[5])
    assert dpz.device_status() == 0


def _random_ranges(rng, N, C):
    """The arena [0, N*C) cut at random segment boundaries of its chunks (a
    range may span chunks), as a shuffled list of (lo, n)."""
    cuts = [c * C + 256 * j for c in range(N) for j in range((C + 255) // 256)] + [N * C]
    cuts = sorted(set(cuts))
    keep = [0] + [x for x in cuts[1:-1] if rng.random() < 0.3] + [N * C]
    ranges = [(a, b - a) for a, b in zip(keep[:-1], keep[1:])]
    rng.shuffle(ranges)
    return ranges


@pytest.mark.parametrize("seed", [2000 + k for k in range(24)])
def test_random_buckets_match_oracle(seed):
    dpz = _dpz()
    w, acc32, _, rng = _case(seed)
    N, C = w.N, w.C
    g, th, m, v, wts = _inputs(w)
    G, T, M, V, W = up(g), up(th), up(m), up(v), up(wts)
    ws = dpz.workspace(w.P, N, DEV)
    nrm = torch.full((1,), -1.0, device=DEV)
    cfg = dpz.make_cfg(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.step, w.clip)
    ranges = _random_ranges(rng, N, C)
    max_ctas = int(rng.choice([0, 1, 152]))
    for lo, n in ranges:
        dpz.dp_reduce_scatter_avg_range(G, N, lo, n, ws=ws, acc32=acc32, max_ctas=max_ctas)
    dpz.dp_grad_norm_finalize(ws, w.P, N, nrm)
    dpz.dp_zero1_update(G, T, M, V, W, N, cfg, ws=ws)
    torch.cuda.synchronize()
    assert dpz.ws_status(ws) == 0
    out = (down(G).reshape(N, w.P), down(T), down(M), down(V), down(W).reshape(N, w.P),
           nrm.item())
    check_step(w, g, th, m, v, wts, out, check_avg=True, acc32=acc32)
    assert dpz.device_status() == 0
