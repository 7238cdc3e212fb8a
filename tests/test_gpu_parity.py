"""GPU parity: every entry point of the C-ABI against the CPU oracle on the same
seeded inputs, at sizes that span several grid-stride tiles with a ragged
tail, plus the edge cases (N = 1, minimal chunks, NaN/Inf, subnormals,
non-power-of-two N, N up to 64)."""
import numpy as np
import pytest
import torch

import inputs as I
import oracle as O

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import gradient_reduction_zero_gb300.dpz as dpz
    from gpu_util import DEV, check_step, down, np_dtype, same_bits, up

# (N, C): C = chunk elements.  2048 elements = one block-iteration of a
# 256-thread block; C = 3_000_016 makes every thread loop several times.
SHAPES = [(1, 8), (1, 4104), (2, 8), (2, 2056), (3, 1000), (4, 1024), (4, 6152),
          (5, 2000), (7, 776), (8, 12344), (16, 520), (64, 72), (4, 3_000_016)]


def rand_grads(N, C, gdt, seed, sigma=1.0):
    w = I.TINY.with_(N=N, P=N * C, gdtype=gdt, grad=I.Dist(I.NORMAL, sigma), grad_seed=seed)
    return I.arena_host(w)


def oracle_rs(g):
    a = g.copy()
    O.ring_reduce_scatter(a)
    O.average_owned(a)
    return a


# ----------------------------------------------------------- reduce-scatter

@pytest.mark.parametrize("N,C", SHAPES)
@pytest.mark.parametrize("gdt", ["f32", "bf16"])
def test_reduce_scatter_avg(N, C, gdt):
    g = rand_grads(N, C, gdt, seed=N * 100 + C % 97)
    ref = oracle_rs(g)
    G = up(g)
    dpz.dp_reduce_scatter_avg(G, N)
    out = down(G)
    for c in range(N):
        for r in range(N):
            sl = slice(c * C, (c + 1) * C)
            want = ref[c, sl] if r == c else g[r, sl]       # other chunks untouched
            assert same_bits(out[r, sl], want), (r, c)


@pytest.mark.parametrize("N,C", SHAPES)
@pytest.mark.parametrize("gdt", ["f32", "bf16"])
def test_allreduce_avg(N, C, gdt):
    g = rand_grads(N, C, gdt, seed=7 + N)
    ref = g.copy()
    O.ring_allreduce_avg(ref)
    G = up(g)
    dpz.dp_allreduce_avg(G, N)
    assert same_bits(down(G), ref)


@pytest.mark.parametrize("N,C", [(1, 8), (2, 2056), (4, 6152), (8, 776), (64, 72)])
@pytest.mark.parametrize("wdt", ["f32", "bf16"])
def test_allgather(N, C, wdt):
    w = rand_grads(N, C, wdt, seed=3)
    ref = w.copy()
    O.ring_allgather(ref)
    W = up(w)
    dpz.dp_allgather(W, N)
    assert same_bits(down(W), ref)


# ----------------------------------------------------------- norm

@pytest.mark.parametrize("N,C", [(1, 8), (3, 1000), (4, 6152), (8, 12344), (4, 3_000_016)])
@pytest.mark.parametrize("gdt", ["f32", "bf16"])
def test_global_norm(N, C, gdt):
    g = rand_grads(N, C, gdt, seed=11 * N, sigma=1e-3)
    ref = oracle_rs(g)
    onorm, _ = O.clip_scale(O.sumsq_owned(ref), 0.0)
    G = up(g)
    ws = dpz.workspace(N * C, N, DEV)
    nrm = torch.zeros(1, device=DEV)
    dpz.dp_reduce_scatter_avg(G, N)
    dpz.dp_grad_global_norm(G, N, ws, nrm)
    gn = nrm.item()
    assert abs(gn - onorm) <= 1e-6 * onorm
    # the staged norm kernel writes the same per-segment partials as the
    # reduce kernel: the norm of the fused path is the same float
    G2 = up(g)
    nrm2 = torch.zeros(1, device=DEV)
    ws2 = dpz.workspace(N * C, N, DEV)
    T = torch.zeros(N * C, device=DEV)
    W = torch.zeros(N * N * C, dtype=G2.dtype, device=DEV)
    cfg = dpz.make_cfg(1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1e30)   # clip that never triggers
    dpz.dp_zero1_step(G2, T, T.clone(), T.clone(), W, N, cfg, ws=ws2, norm_out=nrm2)
    assert nrm2.item() == gn
    assert dpz.device_status() == 0


# ----------------------------------------------------------- the step

def make_problem(N, C, gdt, wdt, clip, seed, step=1000, gsigma=1e-3):
    w = I.TINY.with_(N=N, P=N * C, gdtype=gdt, wdtype=wdt, clip=clip,
                     grad=I.Dist(I.NORMAL_TAIL, gsigma), grad_seed=seed,
                     m=I.Dist(I.NORMAL, 1e-4), v=I.Dist(I.ABS_NORMAL, 1e-6),
                     lr=1.5e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, step=step)
    g = I.arena_host(w)
    th, m, v = (I.state_host(w, k) for k in ("master", "m", "v"))
    wts = np.full((N, w.P), 0x7F7F if wdt == "bf16" else 3.0, dtype=np_dtype(wdt))
    return w, g, th, m, v, wts


def run_gpu_step(w, g, th, m, v, wts, store_avg=True, want_norm=True, fused=True, acc32=False):
    G, T, M, V, W = up(g), up(th), up(m), up(v), up(wts)
    ws = dpz.workspace(w.P, w.N, DEV)
    nrm = torch.full((1,), -1.0, device=DEV)
    cfg = dpz.make_cfg(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.step, w.clip,
                       store_avg=store_avg)
    if fused:
        dpz.dp_zero1_step(G, T, M, V, W, w.N, cfg, ws=ws, norm_out=nrm if want_norm else None,
                          acc32=acc32)
    else:
        dpz.dp_reduce_scatter_avg(G, w.N, acc32=acc32)
        if w.clip > 0 or want_norm:
            dpz.dp_grad_global_norm(G, w.N, ws, nrm)
        dpz.zero1_adamw_step(G, T, M, V, W, w.N, cfg, ws=ws)
        dpz.dp_allgather(W, w.N)
    torch.cuda.synchronize()
    if w.clip > 0 or want_norm:          # a finalisation ran: no tile was skipped
        assert dpz.ws_status(ws) == 0
    return down(G), down(T), down(M), down(V), down(W), nrm.item()


@pytest.mark.parametrize("store_avg", [False, True])
def test_tiny_workload_as_stated(store_avg):
    """The tiny workload exactly as its recipe states it, inputs unmodified:
    N = 4, P = 4,096, fp32 gradients U(-1, 1) seeded by rank, master
    N(0, 0.02), m = v = 0, t = 1, lr 1e-3, betas (0.9, 0.999), eps 1e-8,
    weight decay 0.1, no clip, bf16 weights.  dp_zero1_step with the norm
    output (the one-block kernel the benchmark times) gives the oracle's bits
    for master, m, v, every weight replica and, with store_avg, the averages;
    without store_avg the gradients are left as they were."""
    w = I.TINY
    assert (w.N, w.P, w.gdtype, w.wdtype, w.clip, w.step) == (4, 4096, "f32", "bf16", 0.0, 1)
    g = I.arena_host(w)
    th, m, v = (I.state_host(w, k) for k in ("master", "m", "v"))
    assert not m.any() and not v.any()
    assert np.abs(g).max() <= 1.0
    wts = np.zeros((w.N, w.P), dtype=np.uint16)
    before = dpz.launch_count()
    out = run_gpu_step(w, g, th, m, v, wts, store_avg=store_avg)
    assert dpz.launch_count() - before == 1
    check_step(w, g, th, m, v, wts, out, check_avg=store_avg)
    if not store_avg:
        assert same_bits(out[0], g)
    assert dpz.device_status() == 0


# N = 24 (fp32 gradients) and N = 48 (bf16) put the N slab tiles of the staged
# step exactly at its shared-memory limit with bf16 weights and just past it
# with fp32 weights, so both sides of that switch run.  N = 32 with C = 1288
# runs three 512-element tiles per chunk, the last one ragged, in every dtype
# pair.
STEP_SHAPES = [(1, 8), (1, 4104), (2, 2056), (3, 1000), (4, 1024), (4, 6152), (5, 2000),
               (8, 12344), (16, 520), (24, 1032), (32, 1288), (48, 264), (64, 72),
               (4, 3_000_016)]


@pytest.mark.parametrize("N,C", STEP_SHAPES)
@pytest.mark.parametrize("gdt,wdt", [("bf16", "bf16"), ("f32", "bf16"), ("f32", "f32"),
                                     ("bf16", "f32")])
@pytest.mark.parametrize("clip", [0.0, 1e-3])
def test_zero1_step(N, C, gdt, wdt, clip):
    w, g, th, m, v, wts = make_problem(N, C, gdt, wdt, clip, seed=N + C % 13)
    out = run_gpu_step(w, g, th, m, v, wts)
    check_step(w, g, th, m, v, wts, out)


@pytest.mark.parametrize("N,C", [(4, 6152), (8, 776), (3, 1000)])
@pytest.mark.parametrize("clip", [0.0, 1e-3])
def test_fused_equals_unfused(N, C, clip):
    """dp_zero1_step is bit-identical to the four separate calls."""
    w, g, th, m, v, wts = make_problem(N, C, "bf16", "bf16", clip, seed=5)
    a = run_gpu_step(w, g, th, m, v, wts, fused=True)
    b = run_gpu_step(w, g, th, m, v, wts, fused=False)
    for x, y in zip(a[:5], b[:5]):
        assert same_bits(x, y)
    assert a[5] == b[5]


@pytest.mark.parametrize("N,C,launches", [(4, 2048, 1), (3, 2816, 2), (4, 1024, 1), (1, 8, 1),
                                           (8, 1024, 1), (8, 1032, 2)])
@pytest.mark.parametrize("gdt", ["f32", "bf16"])
def test_small_step_is_one_launch_and_identical(N, C, launches, gdt):
    """Without clip and with the norm wanted, an arena of at most 32 segments
    runs the step and its norm in one launch (a thread-block cluster); larger ones use the
    fold kernel plus the finalisation.  Both give the four separate calls'
    bits, the norm included."""
    w, g, th, m, v, wts = make_problem(N, C, gdt, "bf16", 0.0, seed=C + N)
    before = dpz.launch_count()
    a = run_gpu_step(w, g, th, m, v, wts, fused=True)
    assert dpz.launch_count() - before == launches
    b = run_gpu_step(w, g, th, m, v, wts, fused=False)
    for x, y in zip(a[:5], b[:5]):
        assert same_bits(x, y)
    assert a[5] == b[5]
    check_step(w, g, th, m, v, wts, a)


@pytest.mark.parametrize("N,segs", [(1, 1), (1, 2), (1, 3), (1, 5), (1, 8), (1, 9), (1, 15),
                                    (1, 17), (1, 24), (1, 25), (1, 31), (1, 32), (2, 7),
                                    (3, 10), (4, 8), (5, 6), (7, 4), (8, 4), (16, 2), (32, 1)])
def test_small_step_every_cluster_shape(N, segs):
    """The one-launch small step spreads 1 to 32 segments over a thread-block
    cluster of up to 8 CTAs (1 to 4 warps each; some warps of the last CTA
    idle).  Every shape gives the four separate calls' bits, the norm
    included, and the oracle's.  Each chunk ends in a ragged segment."""
    C = segs * 256 - 8
    w, g, th, m, v, wts = make_problem(N, C, "bf16", "bf16", 0.0, seed=N * 64 + segs)
    before = dpz.launch_count()
    a = run_gpu_step(w, g, th, m, v, wts, fused=True)
    assert dpz.launch_count() - before == 1
    b = run_gpu_step(w, g, th, m, v, wts, fused=False)
    for x, y in zip(a[:5], b[:5]):
        assert same_bits(x, y)
    assert a[5] == b[5]
    check_step(w, g, th, m, v, wts, a)


def test_prepared_call_equals_plain_call():
    """A prepared step (arguments marshalled once) gives the plain call's
    bits, step after step."""
    w, g, th, m, v, wts = make_problem(4, 6152, "bf16", "bf16", 1e-3, seed=77)
    outs = []
    for prepared in (False, True):
        G, T, M, V, W = up(g), up(th), up(m), up(v), up(wts)
        ws = dpz.workspace(w.P, w.N, DEV)
        nrm = torch.zeros(1, device=DEV)
        cfg = dpz.make_cfg(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.step, w.clip)
        if prepared:
            call = dpz.prepare_zero1_step(G, T, M, V, W, w.N, cfg, ws=ws, norm_out=nrm)
            for _ in range(3):
                call()
        else:
            for _ in range(3):
                dpz.dp_zero1_step(G, T, M, V, W, w.N, cfg, ws=ws, norm_out=nrm)
        torch.cuda.synchronize()
        outs.append([down(x) for x in (G, T, M, V, W)] + [nrm.item()])
    for x, y in zip(outs[0][:5], outs[1][:5]):
        assert same_bits(x, y)
    assert outs[0][5] == outs[1][5]


@pytest.mark.parametrize("store_avg,want_norm", [(False, False), (False, True), (True, False)])
def test_no_clip_variants(store_avg, want_norm):
    N, C = 4, 6152
    w, g, th, m, v, wts = make_problem(N, C, "bf16", "bf16", 0.0, seed=9)
    out = run_gpu_step(w, g, th, m, v, wts, store_avg=store_avg, want_norm=want_norm)
    Gg = out[0]
    if not store_avg:
        assert same_bits(Gg, g)          # gradients left as they were
    if not want_norm:
        assert out[5] == -1.0
    check_step(w, g, th, m, v, wts, out, check_avg=store_avg)


@pytest.mark.parametrize("gdt,wdt", [("bf16", "bf16"), ("f32", "f32"), ("bf16", "f32")])
@pytest.mark.parametrize("N,C", [(4, 3_000_016), (3, 1000), (16, 520)])
def test_staged_update_equals_owner_update_plus_allgather(gdt, wdt, N, C):
    """The clipped step's AdamW + all-gather kernel stages 1024-element tiles
    through shared memory by bulk copies (ragged last tile per chunk, runtime
    and compile-time N): bit-identical to the owner-only update plus the
    separate all-gather, and no bounded wait ran out."""
    w, g, th, m, v, wts = make_problem(N, C, gdt, wdt, 1e-3, seed=17 + N)
    assert dpz.device_status() == 0
    a = run_gpu_step(w, g, th, m, v, wts, fused=True)
    b = run_gpu_step(w, g, th, m, v, wts, fused=False)
    for x, y in zip(a[:5], b[:5]):
        assert same_bits(x, y)
    assert dpz.device_status() == 0
    check_step(w, g, th, m, v, wts, a)


@pytest.mark.parametrize("N,C", [(4, 6152), (3, 1000)])
def test_clip_boundary(N, C):
    """The clip scales only when norm > clip: with clip equal to the norm the
    clipped (three-kernel) step gives the unclipped step's bits; one float
    below the norm it scales, as the oracle does with the same clip."""
    w, g, th, m, v, wts = make_problem(N, C, "bf16", "bf16", 0.0, seed=31)
    base = run_gpu_step(w, g, th, m, v, wts)                  # no clip; its norm
    norm = np.float32(base[5])
    at = w.with_(clip=float(norm))
    out = run_gpu_step(at, g, th, m, v, wts)
    assert out[5] == base[5]
    for x, y in zip(out[1:5], base[1:5]):                    # master, m, v, weights
        assert same_bits(x, y)
    below = w.with_(clip=float(np.nextafter(norm, np.float32(0))))
    out2 = run_gpu_step(below, g, th, m, v, wts)
    assert not same_bits(out2[1], base[1])                   # scaled this time
    check_step(below, g, th, m, v, wts, out2)


def _random_cases(n_cases, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n_cases):
        N = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 11, 16]))
        C = 8 * int(rng.integers(1, 750))                      # 8 .. 5,992 elements
        gdt, wdt = [("bf16", "bf16"), ("f32", "bf16"), ("f32", "f32"), ("bf16", "f32")][
            int(rng.integers(0, 4))]
        clip = float(rng.choice([0.0, 1e-3]))
        acc32 = gdt == "bf16" and bool(rng.integers(0, 2))
        cases.append((N, C, gdt, wdt, clip, acc32, int(rng.integers(0, 1 << 30))))
    return cases


@pytest.mark.parametrize("N,C,gdt,wdt,clip,acc32,seed", _random_cases(32, 2026))
def test_random_shapes(N, C, gdt, wdt, clip, acc32, seed):
    """Seeded random shapes (N up to 16, chunks of 8 to 5,992 elements, so
    segments, tiles and the small-arena path all meet ragged ends), dtype
    pairs, clip and the fp32-accumulating ring: the fused step against the
    oracle, and against the four separate calls bit for bit."""
    w, g, th, m, v, wts = make_problem(N, C, gdt, wdt, clip, seed=seed)
    a = run_gpu_step(w, g, th, m, v, wts, fused=True, acc32=acc32)
    check_step(w, g, th, m, v, wts, a, acc32=acc32)
    b = run_gpu_step(w, g, th, m, v, wts, fused=False, acc32=acc32)
    for x, y in zip(a[:5], b[:5]):
        assert same_bits(x, y)
    assert a[5] == b[5]


@pytest.mark.parametrize("N,C", [(12, 520), (32, 264), (64, 72)])
@pytest.mark.parametrize("clip", [0.0, 1e-3])
def test_large_n_fp32_accumulating_step(N, C, clip):
    """The fp32-accumulating bf16 ring at large N, where the step without clip
    runs the staged kernel with a run-time fold on 1024- (N = 12) or
    512-element tiles (N = 32, 64): against the oracle, and against the four
    separate calls bit for bit."""
    w, g, th, m, v, wts = make_problem(N, C, "bf16", "bf16", clip, seed=N + 7)
    a = run_gpu_step(w, g, th, m, v, wts, fused=True, acc32=True)
    check_step(w, g, th, m, v, wts, a, acc32=True)
    b = run_gpu_step(w, g, th, m, v, wts, fused=False, acc32=True)
    for x, y in zip(a[:5], b[:5]):
        assert same_bits(x, y)
    assert a[5] == b[5]


def test_deterministic():
    w, g, th, m, v, wts = make_problem(8, 12344, "bf16", "bf16", 1e-3, seed=1)
    a = run_gpu_step(w, g, th, m, v, wts)
    b = run_gpu_step(w, g, th, m, v, wts)
    for x, y in zip(a[:5], b[:5]):
        assert same_bits(x, y)
    assert a[5] == b[5]


def test_multi_step_matches_oracle():
    """Three consecutive steps (t = 1, 2, 3) from m = v = 0."""
    N, C = 4, 2056
    w, g, th, m, v, wts = make_problem(N, C, "bf16", "bf16", 0.0, seed=2, step=1)
    m[:] = 0
    v[:] = 0
    G, T, M, V, W = up(g), up(th), up(m), up(v), up(wts)
    To, Mo, Vo, Wo = th.copy(), m.copy(), v.copy(), wts.copy()
    for t in (1, 2, 3):
        wt = w.with_(step=t)
        gt = I.arena_host(wt.with_(grad_seed=10 * t))
        G.copy_(up(gt))
        cfg = dpz.make_cfg(wt.lr, wt.beta1, wt.beta2, wt.eps, wt.weight_decay, t, 0.0)
        dpz.dp_zero1_step(G, T, M, V, W, N, cfg)
        O.zero1_step(gt.copy(), To, Mo, Vo, Wo, O.cfg_from_workload(wt))
    torch.cuda.synchronize()
    assert same_bits(down(T), To) and same_bits(down(M), Mo) and same_bits(down(V), Vo)
    assert same_bits(down(W), Wo)


# ----------------------------------------------------------- edge cases

def test_nan_inf_propagate():
    N, C = 4, 1024
    w, g, th, m, v, wts = make_problem(N, C, "f32", "bf16", 0.0, seed=3)
    g[1, 5] = np.nan
    g[2, C + 7] = np.inf
    g[0, 2 * C + 9] = -np.inf
    g[3, 2 * C + 9] = np.inf          # inf - inf = NaN in the fold
    out = run_gpu_step(w, g, th, m, v, wts)
    check_step(w, g, th, m, v, wts, out)
    assert np.isnan(out[1][5]) and np.isnan(out[1][2 * C + 9])


def test_subnormal_and_zero_gradients():
    N, C = 4, 1024
    w, g, th, m, v, wts = make_problem(N, C, "f32", "f32", 0.0, seed=4)
    g[:, :C] = 0.0
    g[:, C:2 * C] = np.float32(1e-41)          # subnormal; the average underflows further
    g[:, 2 * C:2 * C + 8] = np.float32(-3e-45)
    out = run_gpu_step(w, g, th, m, v, wts)
    check_step(w, g, th, m, v, wts, out)
    bg = O.f32_to_bf16(g)
    out = run_gpu_step(w.with_(gdtype="bf16"), bg, th, m, v, wts)
    check_step(w.with_(gdtype="bf16"), bg, th, m, v, wts, out)


def test_guard_bands_untouched():
    """Bytes just outside every buffer keep their canary values."""
    N, C = 4, 2056
    w, g, th, m, v, wts = make_problem(N, C, "bf16", "bf16", 1e-3, seed=6)
    pad = 4096

    def guarded(a):
        flat = a.reshape(-1)
        buf = np.full(flat.size + 2 * pad, 0x5A5A if a.dtype == np.uint16 else 1234.5,
                      dtype=a.dtype)
        buf[pad:pad + flat.size] = flat
        return up(buf)

    srcs = (g, th, m, v, wts)
    bufs = [guarded(x) for x in srcs]
    views = [b[pad:-pad].view(x.shape) for b, x in zip(bufs, srcs)]
    ws = dpz.workspace(w.P, N, DEV)
    cfg = dpz.make_cfg(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.step, w.clip)
    dpz.dp_zero1_step(*views, N, cfg, ws=ws)
    torch.cuda.synchronize()
    for b, x in zip(bufs, srcs):
        canary = 0x5A5A if x.dtype == np.uint16 else np.float32(1234.5)
        hb = down(b)
        assert np.all(hb[:pad] == canary) and np.all(hb[-pad:] == canary)


def test_misaligned_tensor_is_refused():
    g = torch.zeros(4 * 1024 + 1, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(dpz.DpzError) as e:
        dpz.dp_reduce_scatter_avg(g[1:], 4)
    assert e.value.code == dpz.ERR_ALIGN


def test_device_generator_matches_host():
    """The inputs the GPU tests and the bench generate on the device are the
    oracle's inputs, bit for bit."""
    for w in (I.GPT2_1P5B.with_(P=4 * 65536), I.TINY):
        t = torch.empty(w.N * w.P, dtype=torch.bfloat16 if w.gdtype == "bf16" else torch.float32,
                        device=DEV)
        I.fill_grads_device(w, t)
        for which in ("master", "m", "v"):
            s = torch.empty(w.P, dtype=torch.float32, device=DEV)
            I.fill_state_device(w, which, s)
            assert np.array_equal(down(s), I.state_host(w, which))
        torch.cuda.synchronize()
        assert np.array_equal(down(t).reshape(w.N, w.P), I.arena_host(w))


def test_profiling_and_launch_count():
    N, C = 4, 6152
    w, g, th, m, v, wts = make_problem(N, C, "bf16", "bf16", 1e-3, seed=8)
    before = dpz.launch_count()
    dpz.profile_start(64)
    run_gpu_step(w, g, th, m, v, wts)
    stats = dpz.profile_stop()
    assert dpz.launch_count() - before == 3
    assert set(stats) == {"dpz_rs_avg_sumsq", "dpz_norm_finalize", "dpz_adamw_bcast"}
    assert all(n == 1 and ms > 0 for n, ms in stats.values())


# ----------------------------------------------------------- fp32-accumulating bf16 ring

@pytest.mark.parametrize("N,C", SHAPES)
def test_acc32_reduce_scatter(N, C):
    g = rand_grads(N, C, "bf16", seed=5 * N + 1)
    ref = g.copy()
    O.reduce_scatter_avg(ref, acc32=True)
    G = up(g)
    dpz.dp_reduce_scatter_avg(G, N, acc32=True)
    out = down(G)
    for c in range(N):
        sl = slice(c * C, (c + 1) * C)
        for r in range(N):
            want = ref[c, sl] if r == c else g[r, sl]
            assert same_bits(out[r, sl], want), (r, c)


@pytest.mark.parametrize("N,C", [(1, 8), (2, 2056), (3, 1000), (4, 6152), (8, 12344), (64, 72)])
def test_acc32_allreduce(N, C):
    g = rand_grads(N, C, "bf16", seed=9 + N)
    ref = g.copy()
    O.ring_allreduce_avg(ref, acc32=True)
    G = up(g)
    dpz.dp_allreduce_avg(G, N, acc32=True)
    assert same_bits(down(G), ref)


@pytest.mark.parametrize("N,C", [(1, 4104), (3, 1000), (4, 6152), (8, 12344), (16, 520)])
@pytest.mark.parametrize("wdt", ["bf16", "f32"])
@pytest.mark.parametrize("clip", [0.0, 1e-3])
def test_acc32_zero1_step(N, C, wdt, clip):
    w, g, th, m, v, wts = make_problem(N, C, "bf16", wdt, clip, seed=2 * N + 3)
    out = run_gpu_step(w, g, th, m, v, wts, acc32=True)
    check_step(w, g, th, m, v, wts, out, acc32=True)


@pytest.mark.parametrize("clip", [0.0, 1e-3])
def test_acc32_fused_equals_unfused(clip):
    w, g, th, m, v, wts = make_problem(4, 6152, "bf16", "bf16", clip, seed=12)
    a = run_gpu_step(w, g, th, m, v, wts, fused=True, acc32=True)
    b = run_gpu_step(w, g, th, m, v, wts, fused=False, acc32=True)
    for x, y in zip(a[:5], b[:5]):
        assert same_bits(x, y)
    assert a[5] == b[5]


def test_resume_from_saved_state():
    """The library keeps no state: saving master/m/v/weights and the step
    counter, then continuing from fresh buffers, equals running on."""
    N, C = 4, 2056
    w, g, th, m, v, wts = make_problem(N, C, "bf16", "bf16", 1e-3, seed=21, step=1)
    m[:] = 0
    v[:] = 0
    grads = [I.arena_host(w.with_(grad_seed=100 * t)) for t in (1, 2, 3)]

    def run(state, steps):
        T, M, V, W = (up(x) for x in state)
        ws = dpz.workspace(w.P, N, DEV)
        for t in steps:
            cfg = dpz.make_cfg(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, t, w.clip)
            dpz.dp_zero1_step(up(grads[t - 1]), T, M, V, W, N, cfg, ws=ws)
        torch.cuda.synchronize()
        return [down(x) for x in (T, M, V, W)]

    straight = run((th, m, v, wts), (1, 2, 3))
    saved = run((th, m, v, wts), (1, 2))            # a checkpoint after step 2
    resumed = run(saved, (3,))
    for a, b in zip(straight, resumed):
        assert same_bits(a, b)
