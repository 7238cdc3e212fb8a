"""Helpers for the GPU parity tests: host<->device copies of oracle-format
arrays and the comparison rules (bit-exact where the arithmetic is the same
sequence of IEEE operations; the stated tolerances otherwise)."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O

DEV = torch.device("cuda:0")


def up(a: np.ndarray, device=DEV) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return t.view(torch.bfloat16) if a.dtype == np.uint16 else t


def down(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def np_dtype(dt: str):
    return np.uint16 if dt == "bf16" else np.float32


def f32_view(a: np.ndarray) -> np.ndarray:
    return O.bf16_to_f32(a) if a.dtype == np.uint16 else a


def same_bits(a: np.ndarray, b: np.ndarray) -> bool:
    """Bitwise equality, except that any NaN matches any NaN."""
    if a.shape != b.shape or a.dtype != b.dtype:
        return False
    fa, fb = f32_view(a), f32_view(b)
    na, nb = np.isnan(fa), np.isnan(fb)
    if not np.array_equal(na, nb):
        return False
    return np.array_equal(a[~na], b[~nb])


def ulp_distance_bf16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 units in the last place (ordered integer space)."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), x + 0x8000)
    return np.abs(ordered(a) - ordered(b))


def assert_weights(gpu: np.ndarray, ref: np.ndarray, exact: bool):
    if exact or gpu.dtype == np.float32:
        if exact:
            assert same_bits(gpu, ref), "weights differ"
        return
    fa = O.bf16_to_f32(gpu)
    nan = np.isnan(fa)
    assert np.array_equal(nan, np.isnan(O.bf16_to_f32(ref)))
    d = ulp_distance_bf16(gpu[~nan], ref[~nan])
    assert d.max(initial=0) <= 1, f"bf16 weights differ by {d.max()} ulp"


def state_tolerances(avg_f32, scale, th0, m0, v0, m1, v1, cfg, rtol=1e-6):
    """Per-element error budgets of rtol relative to the terms of each update
    (the operands' magnitudes), so that cancellation does not turn a tiny
    difference in the clip scale into a large relative error."""
    b1, b2, lr, eps, wd = cfg.beta1, cfg.beta2, cfg.lr, cfg.eps, cfg.weight_decay
    gs = avg_f32.astype(np.float64) * scale
    tm = rtol * (b1 * np.abs(m0) + (1 - b1) * np.abs(gs))
    tv = rtol * (b2 * np.abs(v0) + (1 - b2) * gs * gs) + 1e-45
    bc1, bc2 = O.bias_corrections(cfg)
    upd = (m1.astype(np.float64) / bc1) / (np.sqrt(np.abs(v1.astype(np.float64)) / bc2) + eps)
    tt = rtol * (np.abs(th0) + lr * (np.abs(upd) + wd * np.abs(th0))) + 1e-45
    return tm, tv, tt


def assert_close_tol(gpu, ref, tol, what):
    g, r = gpu.astype(np.float64), ref.astype(np.float64)
    nan = np.isnan(r)
    assert np.array_equal(np.isnan(g), nan), f"{what}: NaN positions differ"
    bad = np.abs(g[~nan] - r[~nan]) > tol[~nan]
    assert not bad.any(), f"{what}: {bad.sum()} elements outside tolerance"


def check_step(w, g, th, m, v, wts, out, check_avg=True, acc32=False):
    """One GPU step `out` = (grads, master, m, v, weights, norm) against the
    oracle's zero1_step on the same inputs: the averaged owner chunks bit for
    bit (check_avg), the norm within relative 1e-6 (norm < 0: not asked for),
    and master/m/v and the weights bit for bit when the two norms are the same
    float (always without clip), else within the stated tolerances."""
    Gg, Tg, Mg, Vg, Wg, gnorm = out
    cfg = O.cfg_from_workload(w)
    G, T, M, V, W = g.copy(), th.copy(), m.copy(), v.copy(), wts.copy()
    onorm, oscale, _, _ = O.zero1_step(G, T, M, V, W, cfg, acc32=acc32)
    C = w.C
    if gnorm >= 0:
        assert abs(gnorm - onorm) <= 1e-6 * onorm, (gnorm, onorm)
    if check_avg:
        for c in range(w.N):
            sl = slice(c * C, (c + 1) * C)
            assert same_bits(Gg[c, sl], G[c, sl]), f"averaged chunk {c}"
    exact = w.clip <= 0 or gnorm == onorm
    if exact:
        assert same_bits(Tg, T) and same_bits(Mg, M) and same_bits(Vg, V)
        assert same_bits(Wg, W)
        return
    avg = np.concatenate([f32_view(G[c, c * C:(c + 1) * C]) for c in range(w.N)])
    tm, tv, tt = state_tolerances(avg, oscale, th, m, v, M, V, cfg)
    assert_close_tol(Mg, M, tm, "m")
    assert_close_tol(Vg, V, tv, "v")
    assert_close_tol(Tg, T, tt, "master")
    if Wg.dtype == np.uint16:
        assert_weights(Wg, W, exact=False)
    else:
        for r in range(w.N):
            assert_close_tol(Wg[r], W[r], tt, "weights")
