"""Pins for the CPU oracle: each test ties the oracle to something other than
itself — values the pages print, closed forms, library routines, invariants the
pages state, or brute force on tiny inputs."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O

CHUNK = {"a": 0, "b": 1, "c": 2}


# ----------------------------------------------------------------- the ring

def test_ring_n3_table(golden):
    """Lab 09 §1: the N = 3 table, row by row.  Rank r's value is 2**r, so a
    chunk's value is the bitmask of the contributions it holds."""
    rows = golden("ring_n3_table.txt")
    N, width = 3, 2
    base = np.zeros((N, N * width), dtype=np.float32)
    for r in range(N):
        base[r, :] = float(2 ** r)
    for phase, step, rank, chunk, contrib, _frm in rows:
        step, rank = int(step), int(rank)
        c = CHUNK[chunk]
        want = sum(2 ** int(k) for k in contrib.split(","))
        a = base.copy()
        if phase == "rs":
            O.ring_reduce_scatter(a, rho=0, steps=step + 1)
        else:
            O.ring_reduce_scatter(a, rho=0, steps=N - 1)
            O.ring_allgather(a, rho=0, steps=step + 1)
        got = a[rank, c * width:(c + 1) * width]
        assert np.all(got == want), (phase, step, rank, chunk, got, want)
    # "afterwards rank r owns the finished chunk (r + 1) mod N" (Lab 09 Tips)
    for r in range(N):
        assert O.owner((r + 1) % N, N, rho=0) == r


def test_ring_n3_table_untouched_chunks(golden):
    """In reduce-scatter step 0 only the chunk named in the table changes at
    each rank; the other two keep the rank's own contribution."""
    N, width = 3, 1
    a = np.array([[float(2 ** r)] * N for r in range(N)], dtype=np.float32)
    O.ring_reduce_scatter(a, rho=0, steps=1)
    changed = {0: "c", 1: "a", 2: "b"}
    for r in range(N):
        for name, c in CHUNK.items():
            if name != changed[r]:
                assert a[r, c] == 2 ** r


@pytest.mark.parametrize("rho", [0, 1])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8])
def test_ring_every_rank_has_the_full_sum(N, rho):
    """Lab 09 'What to implement' row 1: every rank ends with the elementwise
    sum (integer-valued float64, so every order is exact)."""
    rng = np.random.default_rng(N * 10 + rho)
    a = rng.integers(-1000, 1000, size=(N, 64 * N)).astype(np.float64)
    want = a.sum(axis=0)
    O.ring_reduce_scatter(a, rho=rho)
    O.ring_allgather(a, rho=rho)
    for r in range(N):
        assert np.array_equal(a[r], want)


@pytest.mark.parametrize("rho", [0, 1])
@pytest.mark.parametrize("N", [4, 2, 3, 8])
def test_ring_contribution_counts(N, rho):
    """13.5 Multi-GPU from First Principles, 13.5.3 and Figure 13.5.3: with
    every rank's input 1, a cell holds the number of the N contributions its
    chunk has.  Each reduce-scatter step moves one chunk per link, so each rank
    gains exactly one cell, which holds one more contribution than the
    sender's copy: after step t a rank's counts are 2..t+2 and N-1-t ones.
    After the phase every device owns one full chunk (N), a different chunk per
    device.  Each all-gather step then completes one more cell per rank, until
    all N x N cells are full."""
    width = 3
    ones = np.ones((N, N * width), dtype=np.float64)

    def counts(a):
        cells = a.reshape(N, N, width)
        assert np.all(cells == cells[:, :, :1])          # a chunk moves as a whole
        return cells[:, :, 0].astype(int)

    prev = counts(ones)
    for t in range(N - 1):
        a = ones.copy()
        sent = O.ring_reduce_scatter(a, rho=rho, steps=t + 1)
        cur = counts(a)
        assert np.all(sent == (t + 1) * width * 8)          # one chunk per link per step
        for r in range(N):
            assert sorted(cur[r]) == [1] * (N - 1 - t) + list(range(2, t + 3))
            assert np.sum(cur[r] != prev[r]) == (1 if N > 1 else 0)
        prev = cur
    full = [int(np.flatnonzero(prev[r] == N)[0]) for r in range(N)]
    assert all(np.sum(prev[r] == N) == 1 for r in range(N))
    assert sorted(full) == list(range(N))                   # a different chunk per device
    for r in range(N):
        assert O.owner(full[r], N, rho=rho) == r
    for t in range(N - 1):
        a = ones.copy()
        O.ring_reduce_scatter(a, rho=rho)
        O.ring_allgather(a, rho=rho, steps=t + 1)
        cur = counts(a)
        for r in range(N):
            assert np.sum(cur[r] == N) == t + 2
    assert np.all(cur == N)


def test_owner_with_rotation_one_is_zero1_shard_offset():
    """A4 Part 2: rank r's shard starts at r * shard_size, so with rho = 1
    rank c owns chunk c."""
    for N in range(1, 17):
        for c in range(N):
            assert O.owner(c, N, rho=1) == c


@pytest.mark.parametrize("N,ring,naive", [(2, 512, 512), (4, 768, 1536), (8, 896, 3584)])
def test_ring_bytes_match_the_lab(golden, N, ring, naive):
    """Lab 09 §1: 64 float64 values; ring sends 512/768/896 bytes per rank,
    rank 0 of gather-then-broadcast receives 512/1536/3584."""
    table = {int(n): (int(s), int(r)) for n, s, r in golden("ring_bytes.txt")}
    assert table[N] == (ring, naive)
    a = np.ones((N, 64), dtype=np.float64)
    sent = O.ring_allreduce_avg(a.copy())
    assert np.all(sent == ring)
    recv = O.star_allreduce(a.copy())
    assert recv[0] == naive


@pytest.mark.parametrize("N", [2, 3, 4, 8])
@pytest.mark.parametrize("dt,es", [(np.float32, 4), (np.uint16, 2)])
def test_ring_bytes_general(N, dt, es):
    """13.5 Multi-GPU from First Principles, Eq. 13.5.1: 2(k-1)/k * S per
    device; each phase moves (N-1)/N * S."""
    P = 8 * N * 5
    a = np.zeros((N, P), dtype=dt)
    srs = O.ring_reduce_scatter(a, rho=1)
    sag = O.ring_allgather(a, rho=1)
    S = P * es
    assert np.all(srs == (N - 1) * S // N)
    assert np.all(srs + sag == 2 * (N - 1) * S // N)


def test_ring_n1_is_a_no_op():
    a = np.arange(16, dtype=np.float32).reshape(1, 16)
    b = a.copy()
    sent = O.ring_allreduce_avg(b)
    assert np.array_equal(a, b) and sent[0] == 0


# ------------------------------------------------------- fold order / rounding

def test_fold_order_follows_the_table():
    """Lab 09 §1 table, rho = 0: chunk a is built as a1 + a0 at rank 1, then
    a2 + (a0 + a1) at rank 2.  With a0 = 2**24, a1 = 1, a2 = -2**24 the fp32
    sum (a0 + a1) + a2 is 0 (2**24 + 1 rounds to 2**24); any other first pair
    gives 1."""
    big = float(2 ** 24)
    for c in range(3):
        x = np.zeros((3, 3), dtype=np.float32)
        first, second, last = c, (c + 1) % 3, (c + 2) % 3
        x[first, c], x[second, c], x[last, c] = big, 1.0, -big
        O.ring_reduce_scatter(x, rho=0)
        assert x[O.owner(c, 3, rho=0), c] == 0.0
        # the same values with the last contribution first give 1
        y = np.zeros((3, 3), dtype=np.float32)
        y[last, c], y[second, c], y[first, c] = big, 1.0, -big
        O.ring_reduce_scatter(y, rho=0)
        assert y[O.owner(c, 3, rho=0), c] == 1.0


def test_fold_order_rotation_one():
    """rho = 1: chunk c starts at rank c+1, then c+2, ..., and ends at its
    owner c.  Same construction as above."""
    big = float(2 ** 24)
    N = 4
    for c in range(N):
        x = np.zeros((N, N), dtype=np.float32)
        x[(c + 1) % N, c] = big
        x[(c + 2) % N, c] = 1.0
        x[(c + 3) % N, c] = -big
        O.ring_reduce_scatter(x, rho=1)
        assert x[c, c] == 0.0


def _exact_avg_f32(vals, N):
    s = sum(Fraction(float(v)) for v in vals)
    return np.float32(float(s / N))


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 7, 8])
def test_reduce_integer_valued_is_exact(N):
    """Brute force: integer-valued inputs make every partial sum exact, so the
    averaged chunk is the correctly rounded exact mean, in fp32 and bf16."""
    rng = np.random.default_rng(N)
    C = 16
    vals = rng.integers(-16, 17, size=(N, N * C)).astype(np.float32)
    a32 = vals.copy()
    O.ring_reduce_scatter(a32, rho=1)
    O.average_owned(a32, rho=1)
    abf = O.f32_to_bf16(vals)
    O.ring_reduce_scatter(abf, rho=1)
    O.average_owned(abf, rho=1)
    for c in range(N):
        for i in range(C):
            e = c * C + i
            want = _exact_avg_f32(vals[:, e], N)
            assert a32[c, e] == want
            want_bf = torch.tensor([want]).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF
            assert int(abf[c, e]) == want_bf


@pytest.mark.parametrize("N", [2, 3, 4, 8])
def test_reduce_within_rounding_bound_of_exact_sum(N):
    """Random fp32 inputs: the ring's sum is within (N-1) u sum|x| of the exact
    sum (u = 2**-24); bf16 within (N-1) 2**-8 sum|x|."""
    rng = np.random.default_rng(100 + N)
    C = 32
    x = rng.standard_normal((N, N * C)).astype(np.float32)
    for dt, u in ((np.float32, 2.0 ** -24), (np.uint16, 2.0 ** -8)):
        a = x.copy() if dt == np.float32 else O.f32_to_bf16(x)
        xin = a.astype(np.float64) if dt == np.float32 else O.bf16_to_f32(a).astype(np.float64)
        O.ring_reduce_scatter(a, rho=1)
        got = a.astype(np.float64) if dt == np.float32 else O.bf16_to_f32(a).astype(np.float64)
        for c in range(N):
            sl = slice(c * C, (c + 1) * C)
            exact = np.array([float(sum(Fraction(float(v)) for v in xin[:, e]))
                              for e in range(c * C, (c + 1) * C)])
            bound = (N - 1) * u * np.abs(xin[:, sl]).sum(axis=0) * 1.0000001
            assert np.all(np.abs(got[c, sl] - exact) <= bound)


@pytest.mark.parametrize("N", [2, 3, 5, 8])
def test_reduce_equals_left_fold_in_ring_order(N):
    """The message-passing simulation equals a direct left fold of the ranks in
    order c+1, c+2, ..., c (mod N), one rounding per hop."""
    rng = np.random.default_rng(7 * N)
    C = 8
    x = rng.standard_normal((N, N * C)).astype(np.float32)
    xb = O.f32_to_bf16(x)
    a, b = x.copy(), xb.copy()
    O.ring_reduce_scatter(a, rho=1)
    O.ring_reduce_scatter(b, rho=1)
    xbf = torch.from_numpy(O.bf16_to_f32(xb))
    for c in range(N):
        sl = slice(c * C, (c + 1) * C)
        acc = x[(c + 1) % N, sl].copy()
        accb = xbf[(c + 1) % N, sl].clone()
        for j in range(2, N + 1):
            r = (c + j) % N
            acc = (acc + x[r, sl]).astype(np.float32)
            accb = (accb + xbf[r, sl]).to(torch.bfloat16).to(torch.float32)
        assert np.array_equal(a[c, sl], acc)
        assert np.array_equal(O.bf16_to_f32(b[c, sl]), accb.numpy())


def test_averaging_identity_least_squares():
    """Lab 09 §2: the mean of 8 equal-shard gradients of 1/2 mean((Xw - y)^2)
    equals the full-batch gradient X^T (Xw - y) / 64."""
    rng = np.random.default_rng(42)
    n, d, N = 64, 5, 8
    X = rng.standard_normal((n, d))
    y = rng.standard_normal(n)
    w = rng.standard_normal(d)
    full = X.T @ (X @ w - y) / n
    P = 8 * N                       # 5 gradient entries, zero padded
    arena = np.zeros((N, P))
    rows = n // N
    for k in range(N):
        Xk, yk = X[k * rows:(k + 1) * rows], y[k * rows:(k + 1) * rows]
        arena[k, :d] = Xk.T @ (Xk @ w - yk) / rows
    O.ring_allreduce_avg(arena, rho=1)
    for r in range(N):
        np.testing.assert_allclose(arena[r, :d], full, rtol=1e-12, atol=1e-14)
        assert np.all(arena[r, d:] == 0.0)
    # the common bugs of Lab 09: a sum instead of an average is N x too large
    summed = np.zeros((N, P))
    for k in range(N):
        Xk, yk = X[k * rows:(k + 1) * rows], y[k * rows:(k + 1) * rows]
        summed[k, :d] = Xk.T @ (Xk @ w - yk) / rows
    O.ring_reduce_scatter(summed, rho=1)
    O.ring_allgather(summed, rho=1)
    np.testing.assert_allclose(summed[0, :d], N * full, rtol=1e-12)


def test_one_step_one_device_vs_two_shards():
    """13.5 Multi-GPU from First Principles, 13.5.2: one step on one device
    with the whole batch and one step on k = 2 devices with half a batch each
    (mean-loss gradients, averaged) differ only by rounding (the pages measure
    about 1e-9).  Here: the ZeRO-1 step at N = 2 on the shards' gradients
    against N = 1 on the full-batch gradient, least squares, AdamW mid-run
    (m, v nonzero, t = 1000) so that the update depends on the gradient's
    size: a sum instead of an average would move it by far more."""
    rng = np.random.default_rng(7)
    n, d, P = 256, 5, 16                              # P: 5 parameters, zero padded
    X = rng.standard_normal((n, d))
    y = rng.standard_normal(n)
    w0 = np.zeros(P, dtype=np.float32)
    w0[:d] = rng.standard_normal(d) * 0.02
    m0 = np.zeros(P, dtype=np.float32)
    v0 = np.zeros(P, dtype=np.float32)
    m0[:d] = rng.standard_normal(d) * 1e-2
    v0[:d] = np.abs(rng.standard_normal(d)) * 1e-3
    w = w0[:d].astype(np.float64)

    def grad(rows):
        g = np.zeros(P, dtype=np.float32)
        Xk, yk = X[rows], y[rows]
        g[:d] = (Xk.T @ (Xk @ w - yk) / len(yk)).astype(np.float32)
        return g

    cfg = O.cfg_of(1e-3, 0.9, 0.999, 1e-8, 0.1, 1000)

    def step(arena):
        N = arena.shape[0]
        th, m, v = w0.copy(), m0.copy(), v0.copy()
        O.zero1_step(arena, th, m, v, np.zeros((N, P), dtype=np.uint16), cfg)
        return th

    one = step(grad(slice(0, n))[None, :].copy())
    two = step(np.stack([grad(slice(0, n // 2)), grad(slice(n // 2, n))]))
    delta = np.abs(one.astype(np.float64) - two.astype(np.float64))
    assert delta.max() <= 1e-8, delta.max()
    assert np.all(two[d:] == 0.0) and np.all(one[d:] == 0.0)
    # the common bug: the sum of the shard gradients instead of their mean
    summed = np.stack([grad(slice(0, n // 2)), grad(slice(n // 2, n))]) * 2
    bad = step(summed)
    assert np.abs(bad.astype(np.float64) - one.astype(np.float64)).max() > 1e-5


# ------------------------------------------------------------------ bf16

def test_bf16_rounding_matches_torch():
    """The oracle's float->bf16 rounding against torch's CPU conversion
    (round to nearest even) on random bit patterns and edge cases."""
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    edge = np.array([0x00000000, 0x80000000, 0x3F808000, 0x3F818000, 0x3F80FFFF,
                     0x3F807FFF, 0x7F7FFFFF, 0xFF7FFFFF, 0x7F800000, 0xFF800000,
                     0x00000001, 0x00008000, 0x00018000, 0x007FFFFF, 0x7FC00000,
                     0x7F800001, 0xFFFFFFFF], dtype=np.uint32)
    bits = np.concatenate([bits, edge])
    x = bits.view(np.float32)
    ours = O.f32_to_bf16(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(np.isnan(O.bf16_to_f32(ours[nan])))


# ------------------------------------------------------------------ AdamW

def _cfg(lr=1e-3, b1=0.9, b2=0.999, eps=1e-8, wd=0.1, t=1, clip=0.0):
    return O.cfg_of(lr, b1, b2, eps, wd, t, clip)


def test_adamw_first_step_closed_form(golden):
    rows = np.array([[float(v) for v in r] for r in golden("adamw_t1_closed_form.txt")])
    th = rows[:, 0].astype(np.float32)
    g = rows[:, 1].astype(np.float32)
    m = np.zeros_like(th)
    v = np.zeros_like(th)
    O.adamw(th, m, v, g, _cfg())
    lr = 1e-3
    tol = 1e-6 * (np.abs(rows[:, 0]) + lr)
    assert np.all(np.abs(th.astype(np.float64) - rows[:, 2]) <= tol)


def test_adamw_closed_form_fixture_is_its_script_output():
    """The stored closed-form values are what the committed generator writes
    (exact rational arithmetic, no oracle, no CUDA)."""
    import importlib.util
    import os
    from conftest import GOLDEN
    path = os.path.join(GOLDEN, "make_adamw_t1_closed_form.py")
    spec = importlib.util.spec_from_file_location("_make_adamw_t1", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with open(os.path.join(GOLDEN, "adamw_t1_closed_form.txt")) as f:
        assert f.read().splitlines() == mod.lines()


def test_adamw_first_step_closed_form_random():
    rng = np.random.default_rng(5)
    n = 4096
    th0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = rng.uniform(-1, 1, n).astype(np.float32)
    th, m, v = th0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    O.adamw(th, m, v, g, _cfg())
    lr, eps, wd = 1e-3, 1e-8, 0.1
    g64, t64 = g.astype(np.float64), th0.astype(np.float64)
    want = t64 - lr * (g64 / (np.abs(g64) + eps) + wd * t64)
    assert np.all(np.abs(th - want) <= 1e-6 * (np.abs(t64) + lr))
    # the moments use the fp32 values of the hyperparameters
    omb1 = 1.0 - float(np.float32(0.9))
    omb2 = 1.0 - float(np.float32(0.999))
    np.testing.assert_allclose(m, omb1 * g64, rtol=1e-6)
    np.testing.assert_allclose(v, omb2 * g64 * g64, rtol=1e-6)


def test_adamw_pure_decay():
    """g = 0, m = v = 0: the update is only the decoupled decay
    theta * (1 - lr * wd)."""
    th = np.array([1.0, -3.5, 0.02, 0.0], dtype=np.float32)
    t64 = th.astype(np.float64)
    m = np.zeros(4, np.float32)
    v = np.zeros(4, np.float32)
    O.adamw(th, m, v, np.zeros(4, np.float32), _cfg(lr=6e-4, wd=0.1))
    np.testing.assert_allclose(th, t64 * (1 - 6e-4 * 0.1), rtol=2e-7)
    assert np.all(m == 0) and np.all(v == 0)


@pytest.mark.parametrize("t", [1, 2, 1000])
@pytest.mark.parametrize("gdt", ["f32", "bf16"])
def test_adamw_matches_torch(t, gdt):
    """Against torch.optim.AdamW (CPU, fp32, foreach=False) with the state
    injected: same mathematics, different operation order."""
    rng = np.random.default_rng(t)
    n = 8192
    lr, b1, b2, eps, wd = 1.5e-4, 0.9, 0.95, 1e-8, 0.1
    th0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    if gdt == "bf16":
        gb = O.f32_to_bf16(g)
        g = O.bf16_to_f32(gb)
    m0 = (rng.standard_normal(n) * 1e-4).astype(np.float32) if t > 1 else np.zeros(n, np.float32)
    v0 = np.abs(rng.standard_normal(n) * 1e-6).astype(np.float32) if t > 1 else np.zeros(n, np.float32)
    th, m, v = th0.copy(), m0.copy(), v0.copy()
    O.adamw(th, m, v, gb if gdt == "bf16" else g, _cfg(lr, b1, b2, eps, wd, t))

    p = torch.nn.Parameter(torch.from_numpy(th0.copy()))
    opt = torch.optim.AdamW([p], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd,
                            foreach=False, fused=False)
    p.grad = torch.from_numpy(g.copy())
    if t > 1:
        opt.state[p] = {"step": torch.tensor(float(t - 1)),
                        "exp_avg": torch.from_numpy(m0.copy()),
                        "exp_avg_sq": torch.from_numpy(v0.copy())}
    opt.step()
    st = opt.state[p]
    pt = p.detach().numpy().astype(np.float64)
    assert np.all(np.abs(th - pt) <= 1e-6 * (np.abs(th0) + lr))
    mt = st["exp_avg"].numpy().astype(np.float64)
    vt = st["exp_avg_sq"].numpy().astype(np.float64)
    assert np.all(np.abs(m - mt) <= 1e-6 * (b1 * np.abs(m0) + (1 - b1) * np.abs(g)))
    assert np.all(np.abs(v - vt) <= 1e-6 * (b2 * np.abs(v0) + (1 - b2) * g.astype(np.float64) ** 2) + 1e-30)


def test_adamw_padding_stays_zero():
    th = np.zeros(64, np.float32)
    m = np.zeros(64, np.float32)
    v = np.zeros(64, np.float32)
    O.adamw(th, m, v, np.zeros(64, np.float32), _cfg(t=7))
    assert np.all(th == 0) and np.all(m == 0) and np.all(v == 0)


def test_bias_corrections():
    for b1, b2, t in ((0.9, 0.999, 1), (0.9, 0.95, 1000), (0.9, 0.95, 7)):
        bc1, bc2 = O.bias_corrections(_cfg(b1=b1, b2=b2, t=t))
        assert bc1 == np.float32(1 - float(np.float32(b1)) ** t)
        assert bc2 == np.float32(1 - float(np.float32(b2)) ** t)


# ------------------------------------------------------------- norm / clip

def test_global_norm_matches_numpy_and_torch_clip():
    """Norm of the averaged gradient against numpy's fp64 norm, and the clip
    scale against torch.nn.utils.clip_grad_norm_ (which adds 1e-6 to the
    norm)."""
    rng = np.random.default_rng(11)
    N, C = 4, 2048
    x = (rng.standard_normal((N, N * C)) * 1e-1).astype(np.float32)
    a = x.copy()
    O.ring_reduce_scatter(a, rho=1)
    O.average_owned(a, rho=1)
    avg = np.concatenate([a[c, c * C:(c + 1) * C] for c in range(N)])
    ss = O.sumsq_owned(a, rho=1)
    norm, scale = O.clip_scale(ss, 1.0)
    ref = np.linalg.norm(avg.astype(np.float64))
    assert abs(np.sqrt(ss) - ref) <= 1e-12 * ref
    p = torch.nn.Parameter(torch.zeros(avg.size))
    p.grad = torch.from_numpy(avg.copy())
    tn = torch.nn.utils.clip_grad_norm_([p], max_norm=1.0).item()
    assert abs(norm - tn) <= 1e-6 * tn
    coef = 1.0 / (tn + 1e-6)
    assert norm > 1.0 and abs(scale - coef) <= 1e-6 * coef
    # below the threshold nothing is scaled
    n2, s2 = O.clip_scale(ss, 2 * norm)
    assert s2 == 1.0 and n2 == norm
    # clipping off
    assert O.clip_scale(ss, 0.0)[1] == 1.0


# -------------------------------------------------------- ZeRO-1 == ZeRO-0

def _rand_problem(N, C, gdt, wdt, seed):
    rng = np.random.default_rng(seed)
    P = N * C
    g = (rng.standard_normal((N, P)) * 1e-3).astype(np.float32)
    grads = O.f32_to_bf16(g) if gdt == "bf16" else g
    master = (rng.standard_normal(P) * 0.02).astype(np.float32)
    m = (rng.standard_normal(P) * 1e-4).astype(np.float32)
    v = np.abs(rng.standard_normal(P) * 1e-6).astype(np.float32)
    w = np.zeros((N, P), dtype=np.uint16 if wdt == "bf16" else np.float32)
    return grads, master, m, v, w


@pytest.mark.parametrize("clip", [0.0, 1e-3])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("gdt,wdt", [("bf16", "bf16"), ("f32", "bf16"), ("f32", "f32")])
def test_zero1_equals_zero0_bit_for_bit(N, clip, gdt, wdt):
    """Distributed training (noeira), Gates: ZeRO stages are bit-identical to
    DDP; with clipping only the norm's summation order may differ, and here
    both sum in chunk order, so they stay identical.  Lab 09 §4: stage 1 moves
    the same bytes as plain DP."""
    C = 24
    grads, master, m, v, w = _rand_problem(N, C, gdt, wdt, N * 31 + int(clip > 0))
    cfg = _cfg(1.5e-4, 0.9, 0.95, 1e-8, 0.1, 1000, clip)
    g1, t1, m1, v1, w1 = grads.copy(), master.copy(), m.copy(), v.copy(), w.copy()
    norm1, scale1, srs, sag = O.zero1_step(g1, t1, m1, v1, w1, cfg)
    g0 = grads.copy()
    t0 = np.tile(master, (N, 1))
    m0 = np.tile(m, (N, 1))
    v0 = np.tile(v, (N, 1))
    w0 = w.copy()
    norm0, sent0 = O.zero0_step(g0, t0, m0, v0, w0, cfg)
    assert norm0 == norm1
    if clip > 0:
        assert scale1 < 1.0
    for r in range(N):
        assert np.array_equal(t0[r], t1) and np.array_equal(m0[r], m1)
        assert np.array_equal(v0[r], v1)
        assert np.array_equal(w0[r], w1[r])
        assert np.array_equal(w1[r], w1[0])
    # owner chunks hold the average, identical to ZeRO-0's
    for c in range(N):
        sl = slice(c * C, (c + 1) * C)
        assert np.array_equal(g1[c, sl], g0[c, sl])
    # bytes: reduce-scatter + all-gather of the weights vs one gradient
    # all-reduce; identical when gradient and weight dtypes match
    if gdt == wdt:
        assert np.array_equal(srs + sag, sent0)


def test_zero1_n1_is_plain_adamw():
    """Distributed training (noeira), Gates: at N = 1 the distributed step is
    the plain optimizer step."""
    grads, master, m, v, w = _rand_problem(1, 256, "f32", "f32", 9)
    cfg = _cfg(1e-3, 0.9, 0.999, 1e-8, 0.1, 3)
    t1, m1, v1 = master.copy(), m.copy(), v.copy()
    O.zero1_step(grads.copy(), t1, m1, v1, w, cfg)
    p = torch.nn.Parameter(torch.from_numpy(master.copy()))
    opt = torch.optim.AdamW([p], lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.1,
                            foreach=False)
    p.grad = torch.from_numpy(grads[0].copy())
    opt.state[p] = {"step": torch.tensor(2.0), "exp_avg": torch.from_numpy(m.copy()),
                    "exp_avg_sq": torch.from_numpy(v.copy())}
    opt.step()
    assert np.all(np.abs(t1 - p.detach().numpy()) <= 1e-6 * (np.abs(master) + 1e-3))
    assert np.array_equal(w[0], t1)


def test_zero1_window_equals_whole():
    """Element-wise results depend only on the chunk index: a mini-arena made
    of the same window of every chunk gives the same values, given the whole
    arena's sum of squares."""
    N, C = 4, 64
    grads, master, m, v, w = _rand_problem(N, C, "bf16", "bf16", 77)
    cfg = _cfg(6e-4, 0.9, 0.95, 1e-8, 0.1, 1, 0.01)
    G, T, M, V, W = grads.copy(), master.copy(), m.copy(), v.copy(), w.copy()
    norm, scale, _, _ = O.zero1_step(G, T, M, V, W, cfg)
    a = grads.copy()
    O.ring_reduce_scatter(a)
    O.average_owned(a)
    ss = O.sumsq_owned(a)
    off, wd = 16, 8
    cols = np.concatenate([np.arange(c * C + off, c * C + off + wd) for c in range(N)])
    g2 = np.ascontiguousarray(grads[:, cols])
    t2, m2, v2 = master[cols].copy(), m[cols].copy(), v[cols].copy()
    w2 = np.ascontiguousarray(w[:, cols])
    n2, s2, _, _ = O.zero1_step(g2, t2, m2, v2, w2, cfg, ext_sumsq=ss)
    assert (n2, s2) == (norm, scale)
    assert np.array_equal(t2, T[cols]) and np.array_equal(m2, M[cols])
    assert np.array_equal(v2, V[cols]) and np.array_equal(w2, W[:, cols])


def test_oracle_rejects_bad_arguments():
    a = np.zeros((3, 10), dtype=np.float32)     # P = 10 not divisible by N = 3
    with pytest.raises(ValueError):
        O.ring_reduce_scatter(a)
    grads, master, m, v, w = _rand_problem(2, 8, "f32", "f32", 1)
    with pytest.raises(ValueError):
        O.zero1_step(grads, master, m, v, w, _cfg(t=0))


# ------------------------------------------- bf16 ring with fp32 accumulation

@pytest.mark.parametrize("N", [1, 2, 3, 4, 8])
def test_acc32_integer_valued_is_exact(N):
    """With every partial sum exact, both bf16 rings give the correctly
    rounded exact mean."""
    rng = np.random.default_rng(40 + N)
    C = 16
    vals = rng.integers(-16, 17, size=(N, N * C)).astype(np.float32)
    a = O.f32_to_bf16(vals)
    O.reduce_scatter_avg(a, acc32=True)
    for c in range(N):
        for i in range(C):
            e = c * C + i
            want = _exact_avg_f32(vals[:, e], N)
            want_bf = torch.tensor([want]).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF
            assert int(a[c, e]) == want_bf


@pytest.mark.parametrize("N", [2, 3, 5, 8, 64])
def test_acc32_is_one_rounding_of_the_fp32_fold(N):
    """13.5 Multi-GPU from First Principles, Exercise 8, second variant: the
    inputs are bf16 once, the ring's sum is an fp32 left fold in ring order,
    and the average is rounded to bf16 once."""
    rng = np.random.default_rng(7 * N + 1)
    C = 8
    xb = O.f32_to_bf16(rng.standard_normal((N, N * C)).astype(np.float32))
    xf = O.bf16_to_f32(xb)
    a = xb.copy()
    O.reduce_scatter_avg(a, acc32=True)
    for c in range(N):
        sl = slice(c * C, (c + 1) * C)
        acc = xf[(c + 1) % N, sl].copy()
        for j in range(2, N + 1):
            acc = (acc + xf[(c + j) % N, sl]).astype(np.float32)
        avg = (acc / np.float32(N)).astype(np.float32)
        want = torch.from_numpy(avg).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(a[c, sl], want)


def _bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("N", [3, 7])
def test_acc32_average_is_the_ieee_quotient_near_bf16_ties(N):
    """The average divides (Lab 09 — Parallelism, simulated, §2: sum, then
    divide by N).  A product with RN(1/N) differs from the correctly rounded
    quotient in the last fp32 bit for about a third of the sums, and that
    reaches the bf16 result only where the quotient sits next to a bf16 tie:
    about one sum in 10^5.  So the sums here are searched for exactly those
    cases, each split into three exact bf16 parts placed on the first three
    ranks of its chunk's ring order, so that the fp32 fold reproduces it."""
    rng = np.random.default_rng(100 + N)
    bits = rng.integers(0x3F800000, 0x40000000, 2_000_000, dtype=np.uint32)   # [1, 2)
    s = bits.view(np.float32)
    q_ieee = (s.astype(np.float64) / N).astype(np.float32)
    q_recip = (s * (np.float32(1) / np.float32(N))).astype(np.float32)
    hit = np.nonzero(_bf16_bits(q_ieee) != _bf16_bits(q_recip))[0][:4]
    assert len(hit) >= 2
    C = 8
    x = np.zeros((N, N * C), dtype=np.float32)
    sums = s[hit]
    for e, a in enumerate(sums):
        hi = (np.array([a]).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)[0]
        rem = np.float32(a - hi)
        mid = (np.array([rem]).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)[0]
        lo = np.float32(rem - mid)
        for part in (hi, mid, lo):
            assert O.bf16_to_f32(O.f32_to_bf16(np.array([part], dtype=np.float32)))[0] == part
        assert np.float32(np.float32(hi + mid) + lo) == a
        # chunk 0 is folded in rank order 1, 2, ..., N - 1, 0
        x[1, e], x[2, e], x[3 % N, e] = hi, mid, lo
    xb = O.f32_to_bf16(x)
    O.reduce_scatter_avg(xb, acc32=True)
    for e, a in enumerate(sums):
        exact = Fraction(float(a)) / N
        q = np.float32(float(a) / N)                     # nearest float32 to a / N
        ulp = np.spacing(q)
        assert abs(Fraction(float(q)) - exact) < Fraction(float(ulp)) / 2
        want = _bf16_bits(np.array([q]))[0]
        assert int(xb[0, e]) == int(want)
        assert int(want) != int(_bf16_bits(np.array([q_recip[hit[e]]]))[0])


def test_acc32_differs_from_per_hop_rounding():
    """256 + 1 + 1 in a bf16 ring: per-hop rounding loses both ones (257
    rounds to 256), fp32 accumulation keeps them (258 / 3 = 86)."""
    N = 3
    x = np.zeros((N, N), dtype=np.float32)
    # chunk 0 is folded in rank order 1, 2, 0
    x[1, 0], x[2, 0], x[0, 0] = 256.0, 1.0, 1.0
    xb = O.f32_to_bf16(x)
    hop, acc = xb.copy(), xb.copy()
    O.reduce_scatter_avg(hop)
    O.reduce_scatter_avg(acc, acc32=True)
    assert O.bf16_to_f32(hop[0, 0:1])[0] == np.float32(O.bf16_to_f32(O.f32_to_bf16(
        np.array([256.0 / 3], dtype=np.float32)))[0])
    assert O.bf16_to_f32(acc[0, 0:1])[0] == 86.0


@pytest.mark.parametrize("N", [2, 4, 8])
def test_acc32_bytes(N):
    """fp32 partial sums double the reduce-scatter's message bytes; the
    all-gather still moves bf16 averages."""
    P = 8 * N * 4
    a = np.zeros((N, P), dtype=np.uint16)
    sent = O.reduce_scatter_avg(a.copy(), acc32=True)
    assert np.all(sent == (N - 1) * P * 4 // N)
    both = O.ring_allreduce_avg(a.copy(), acc32=True)
    assert np.all(both == (N - 1) * P * 4 // N + (N - 1) * P * 2 // N)


@pytest.mark.parametrize("clip", [0.0, 1e-3])
@pytest.mark.parametrize("N", [1, 3, 4, 8])
def test_acc32_zero1_equals_zero0(N, clip):
    C = 24
    grads, master, m, v, w = _rand_problem(N, C, "bf16", "bf16", 3 * N + int(clip > 0))
    cfg = _cfg(1.5e-4, 0.9, 0.95, 1e-8, 0.1, 1000, clip)
    g1, t1, m1, v1, w1 = grads.copy(), master.copy(), m.copy(), v.copy(), w.copy()
    n1, _, _, _ = O.zero1_step(g1, t1, m1, v1, w1, cfg, acc32=True)
    g0 = grads.copy()
    t0, m0, v0 = (np.tile(x, (N, 1)) for x in (master, m, v))
    w0 = w.copy()
    N_, P_ = g0.shape
    norm = __import__("ctypes").c_float()
    sent = np.zeros(N, dtype=np.int64)
    rc = O.lib().orc_zero0_step(g0.ctypes.data, t0.ctypes.data, m0.ctypes.data, v0.ctypes.data,
                                w0.ctypes.data, N_, P_, O.BF16_ACC32, O.BF16,
                                __import__("ctypes").byref(cfg),
                                __import__("ctypes").addressof(norm), sent.ctypes.data)
    assert rc == 0 and norm.value == n1
    for r in range(N):
        assert np.array_equal(t0[r], t1) and np.array_equal(w0[r], w1[r])
    # the averages match the standalone reduce-scatter's
    a = grads.copy()
    O.reduce_scatter_avg(a, acc32=True)
    for c in range(N):
        assert np.array_equal(g1[c, c * C:(c + 1) * C], a[c, c * C:(c + 1) * C])
