"""The window sweep that the full-size GPU tests rest on (oracle_windows):
its windows tile every chunk exactly, the per-window oracle reproduces the
whole-arena oracle element for element and sum of squares, and a failing
window stops the sweep with its error."""
import math

import numpy as np
import pytest

import inputs as I
import oracle as O
import oracle_windows as OW


@pytest.mark.parametrize("C", [8, 64, 1 << 20, (1 << 20) + 8, 3 * (1 << 20) - 8, 389_402_800])
def test_windows_tile_each_chunk(C):
    wins = OW.chunk_windows(C)
    assert wins[0][0] == 0
    for (o, w), (o2, _) in zip(wins, wins[1:]):
        assert w == OW.WIDTH and o + w == o2            # contiguous, full-width but the last
    o, w = wins[-1]
    assert 0 < w <= OW.WIDTH and o + w == C
    assert all(w % 8 == 0 for _, w in wins)             # whole 8-element groups


def test_window_sweep_reproduces_the_whole_arena():
    """A small arena swept in windows of 24 elements (ragged last window):
    the windows' oracle steps, given the arena's sum of squares, are the
    whole-arena step's values in every element, and their sums of squares add
    up to the arena's."""
    w = I.TINY.with_(N=3, P=3 * 200, gdtype="bf16", wdtype="bf16",
                     grad=I.Dist(I.NORMAL_TAIL, 1e-2), m=I.Dist(I.NORMAL, 1e-4),
                     v=I.Dist(I.ABS_NORMAL, 1e-6), step=5, clip=1e-3)
    N, P, C = w.N, w.P, w.C
    cfg = O.cfg_from_workload(w)
    g = I.arena_host(w)
    th, m, v = (I.state_host(w, k) for k in ("master", "m", "v"))
    G, T, M, V = g.copy(), th.copy(), m.copy(), v.copy()
    W = np.zeros((N, P), dtype=np.uint16)
    O.zero1_step(G, T, M, V, W, cfg)
    ss = OW.oracle_full_sumsq(w)
    a = g.copy()
    O.reduce_scatter_avg(a)
    assert math.isclose(ss, O.sumsq_owned(a), rel_tol=1e-15)

    def window(o, wd):
        gw = I.window_arena_host(w, o, wd)
        tw = I.window_state_host(w, "master", o, wd)
        mw = I.window_state_host(w, "m", o, wd)
        vw = I.window_state_host(w, "v", o, wd)
        ww = np.zeros((N, N * wd), dtype=np.uint16)
        O.zero1_step(gw, tw, mw, vw, ww, cfg, ext_sumsq=ss)
        cols = np.concatenate([np.arange(c * C + o, c * C + o + wd) for c in range(N)])
        for c in range(N):
            sl = slice(c * wd, (c + 1) * wd)
            assert np.array_equal(gw[c, sl], G[c, cols[sl]])     # the owner's averages
        assert np.array_equal(tw, T[cols]) and np.array_equal(mw, M[cols])
        assert np.array_equal(vw, V[cols]) and np.array_equal(ww, W[:, cols])
        return O.sumsq_owned(gw), o, wd

    res = OW.for_every_window(C, window, width=24)
    assert [r[1] for r in res] == [o for o, _ in OW.chunk_windows(C, 24)]
    assert math.fsum(r[0] for r in res) == pytest.approx(ss, rel=1e-15)


def test_failing_window_stops_the_sweep():
    seen = []

    def window(o, wd):
        seen.append(o)
        if o == 5 * 8:
            raise AssertionError("window 40")
        return o

    with pytest.raises(AssertionError, match="window 40"):
        OW.for_every_window(800, window, width=8)
    assert 5 * 8 in seen
