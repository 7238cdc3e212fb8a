"""The oracle on a full-size arena, window by window on all host threads.

A full-size arena does not fit the oracle's host memory at once, so every
chunk is cut into windows and the oracle runs on one window of every chunk at
a time: window [o, o + w) of chunk c becomes chunk c of a mini-arena
[N][N*w].  Each result of the step depends only on its element's values, its
chunk (the ring order) and, through the clip scale, the global norm, so the
oracle's results on the mini-arena are exactly those of the same elements of
the whole arena, given the whole arena's sum of squares."""
from __future__ import annotations

import math
import os
import threading
from concurrent.futures import ThreadPoolExecutor

import inputs as I
import oracle as O

WIDTH = 1 << 20
THREADS = os.cpu_count() or 4


def chunk_windows(C: int, width: int = WIDTH):
    """(offset, width) of the windows that tile a chunk of C elements."""
    return [(o, min(width, C - o)) for o in range(0, C, width)]


def for_every_window(C: int, fn, width: int = WIDTH):
    """fn(o, wd) on every window of every chunk, on all host threads; the
    results in window order.  After the first failure the windows not yet
    started are skipped and that failure is raised."""
    stop = threading.Event()

    def run(ow):
        if stop.is_set():
            return None
        try:
            return fn(*ow)
        except BaseException:
            stop.set()
            raise

    with ThreadPoolExecutor(max_workers=THREADS) as ex:
        futs = [ex.submit(run, ow) for ow in chunk_windows(C, width)]
        return [f.result() for f in futs]


# The whole arena's sum of squares of the averaged gradient, per workload and
# ring mode: the clipped and the unclipped step of one workload share it.
_SUMSQ: dict = {}


def sumsq_key(w: I.Workload, acc32: bool):
    return (w.name, w.N, w.P, w.gdtype, w.grad, w.grad_seed, acc32)


def remember_sumsq(w: I.Workload, acc32: bool, ss: float) -> None:
    _SUMSQ[sumsq_key(w, acc32)] = ss


def oracle_full_sumsq(w: I.Workload, acc32: bool = False) -> float:
    """The oracle's reduce-scatter, average and sum of squares on every
    window, added with math.fsum (the sum of squares is additive over
    windows)."""
    key = sumsq_key(w, acc32)
    if key not in _SUMSQ:
        def part(o, wd):
            g = I.window_arena_host(w, o, wd)
            O.reduce_scatter_avg(g, acc32=acc32)
            return O.sumsq_owned(g)
        _SUMSQ[key] = math.fsum(for_every_window(w.C, part))
    return _SUMSQ[key]
