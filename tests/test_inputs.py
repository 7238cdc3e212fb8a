"""The seeded input generator: counter-based (any window regenerates the same
values), and the distributions the workload recipes ask for."""
import numpy as np

import inputs as I


def test_windows_regenerate_the_same_values():
    d = I.Dist(I.NORMAL_TAIL, 1e-3)
    whole = I.host_fill("f32", 0, 10000, 3, I.STREAM_GRAD, d)
    part = I.host_fill("f32", 1234, 500, 3, I.STREAM_GRAD, d)
    assert np.array_equal(whole[1234:1734], part)
    other_seed = I.host_fill("f32", 0, 10000, 4, I.STREAM_GRAD, d)
    assert not np.array_equal(whole, other_seed)


def test_uniform_range_and_moments():
    x = I.host_fill("f32", 0, 1 << 20, 0, I.STREAM_GRAD, I.Dist(I.UNIFORM))
    assert x.min() >= -1.0 and x.max() < 1.0
    assert abs(x.mean()) < 5e-3 and abs(x.var() - 1 / 3) < 5e-3
    # 24-bit grid
    assert np.all((x.astype(np.float64) * 2 ** 23) == np.round(x.astype(np.float64) * 2 ** 23))


def test_normal_moments_and_tail():
    n = 1 << 20
    x = I.host_fill("f32", 0, n, 7, I.STREAM_GRAD, I.Dist(I.NORMAL, 1e-3)).astype(np.float64)
    assert abs(x.mean()) < 1e-5 and abs(x.std() - 1e-3) < 1e-5
    kurt = ((x - x.mean()) ** 4).mean() / x.var() ** 2
    assert 2.7 < kurt < 3.1                         # Irwin-Hall(12) ~ 2.9
    t = I.host_fill("f32", 0, n, 7, I.STREAM_GRAD, I.Dist(I.NORMAL_TAIL, 1e-3)).astype(np.float64)
    big = np.abs(t) != np.abs(x)
    assert 0.008 < big.mean() < 0.012               # about 1 % scaled x100
    np.testing.assert_allclose(t[big], 100 * x[big], rtol=1e-6)
    a = I.host_fill("f32", 0, n, 7, I.STREAM_GRAD, I.Dist(I.ABS_NORMAL, 1e-6))
    assert np.all(a >= 0)


def test_bf16_inputs_are_truncated_floats():
    f = I.host_fill("f32", 0, 4096, 1, I.STREAM_GRAD, I.Dist(I.NORMAL, 1e-3))
    b = I.host_fill("bf16", 0, 4096, 1, I.STREAM_GRAD, I.Dist(I.NORMAL, 1e-3))
    assert np.array_equal(b, (f.view(np.uint32) >> 16).astype(np.uint16))


def test_workload_shapes():
    for w in (I.TINY, I.GPT2_124M, I.GPT2_1P5B, I.ALLREDUCE_7B):
        assert w.P % (8 * w.N) == 0
    assert I.GPT2_124M.P == 124_439_808 and I.GPT2_1P5B.P == 1_557_611_200
    assert I.GPT2_1P5B.C == 389_402_800 and I.ALLREDUCE_7B.C == 1_750_000_000
    assert [s for s in I.SWEEP_SIZES][0] == 4096 and I.SWEEP_SIZES[-1] == 1 << 30
    for s in I.SWEEP_SIZES:
        for N in (2, 4, 8):
            w = I.allreduce_sweep(s, N)
            assert w.P % (8 * N) == 0


def test_window_arena_layout():
    w = I.TINY
    mini = I.window_arena_host(w, 100, 16)
    full = I.arena_host(w)
    for c in range(w.N):
        assert np.array_equal(mini[:, c * 16:(c + 1) * 16], full[:, c * w.C + 100:c * w.C + 116])
