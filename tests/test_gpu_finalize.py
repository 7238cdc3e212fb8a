"""The norm finalisation on chains of several partials per thread: its sum of
squares against the exact sum of the partials it read, and the chains that
fall back to fp64 (a first-stage sum that overflows fp32; fp32-subnormal,
inf, NaN and skipped-tile marker partials).

The finalisation adds one fp64 partial per 256-element segment of every chunk
(the partials' order is fixed by P and N).  Each of its blocks takes a
contiguous range of them; each thread adds the terms i, i + 512, ... of its
block's range.  An arena needs more than 512 partials (131,072 elements) for
a thread to get two terms, and more than 917,504 for the loop over batches of
eight terms to run, so the arenas here are of those sizes.

The workspace layout read here is the library's own: a 256-byte header
(sumsq as a double at 0, the norm as a float at 8, the status word at 20),
256 first-stage doubles, then the partials in chunk order from byte 2304."""
import math

import numpy as np
import pytest
import torch

import inputs as I

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
PARTIALS_AT = 256 + 256 * 8


def _dpz():
    import gradient_reduction_zero_gb300.dpz as dpz
    return dpz


def _partials(ws, n):
    return ws[PARTIALS_AT:PARTIALS_AT + 8 * n].view(torch.float64).cpu().numpy()


def _sumsq(ws):
    return float(ws[0:8].view(torch.float64).item())


def _owner_sumsq(G, N, P):
    """fp64 sum of squares of the owner chunks (chunk c of slab c)."""
    C = P // N
    g = G.view(N, P)
    tot = 0.0
    for c in range(N):
        x = g[c, c * C:(c + 1) * C].double()
        tot += float(torch.dot(x, x).item())
    return tot


def _tree32(x):
    """The fixed shuffle tree of one warp (offsets 16, 8, 4, 2, 1; lane 0's
    result) over 32 doubles."""
    x = x.copy()
    for o in (16, 8, 4, 2, 1):
        x[:o] = x[:o] + x[o:2 * o]
    return x[0]


def _block_sum(v):
    """The block-wide sum of one double per thread (512 threads): each warp's
    tree, then warp 0's tree over the 16 warp sums (+0 in the other lanes)."""
    w = np.array([_tree32(v[32 * k:32 * k + 32]) for k in range(len(v) // 32)])
    return _tree32(np.concatenate([w, np.zeros(32 - len(w))]))


def _emulated_sumsq(parts):
    """The finalisation's documented arithmetic, step by step on the host:
    F blocks of 512 threads over contiguous ranges, each thread's chain of
    terms i, i + 512, ... added by Sum2 in fp32 (a TwoSum per term, its error
    added into c; s + c then in fp64), or in plain fp64 when a term is not +0
    or a normal fp32 value or the fp32 sum overflows; the block tree; then the
    sum of the F block sums.  Returns the sum of squares it writes."""
    n = len(parts)
    F = min(256, max(1, (n + 2047) // 2048))
    L = (n + F - 1) // F
    bits = parts.view(np.uint64)
    h, l = (bits >> np.uint64(32)).astype(np.uint32), (bits & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    exp = h >> np.uint32(20)
    normal = (exp >= 897) & (exp <= 1150) & ((l & np.uint32(0x1FFFFFFF)) == 0)
    ok_term = normal | ((h == 0) & (l == 0))
    f32 = parts.astype(np.float32)              # exact for the terms that take this path
    stage1 = np.zeros(F)
    with np.errstate(over="ignore", invalid="ignore"):
        for b in range(F):
            lo, hi = b * L, min(b * L + L, n)
            v = np.zeros(512)
            for t in range(512):
                idx = np.arange(lo + t, hi, 512)
                if len(idx) and ok_term[idx].all():
                    s, c = np.float32(0), np.float32(0)
                    for p in f32[idx]:
                        tt = np.float32(s + p)
                        z = np.float32(tt - s)
                        c = np.float32(c + np.float32(np.float32(s - np.float32(tt - z)) + np.float32(p - z)))
                        s = tt
                    if np.isfinite(s):
                        v[t] = np.float64(s) + np.float64(c)
                        continue
                acc = 0.0
                for p in parts[idx]:
                    acc = acc + p
                v[t] = acc
            stage1[b] = _block_sum(v)
    w = np.zeros(512)
    w[:F] = 0.0 + stage1
    return _block_sum(w)


def _norm(G, N, P):
    dpz = _dpz()
    ws = dpz.workspace(P, N, DEV)
    nrm = torch.full((1,), -1.0, device=DEV)
    dpz.dp_grad_global_norm(G, N, ws, nrm)
    torch.cuda.synchronize()
    n = N * ((P // N + 255) // 256)
    return ws, nrm.item(), n


def _wide(w, G):
    """Gradients N(0, 1) scaled by 2^k, k in [-30, 30] varying with the
    element index: segment sums of squares spread over 2^-60 .. 2^60."""
    I.fill_grads_device(w, G)
    idx = torch.arange(G.numel(), device=DEV, dtype=torch.int64)
    k = ((idx // 1000) * 7919 % 61 - 30).to(torch.float32)
    G.mul_(torch.exp2(k).to(G.dtype))


@pytest.mark.parametrize("N,C,gdt", [
    (1, 300_000_000, "bf16"),   # 1.17 M partials: 256 blocks, batches of eight terms and a tail
    (4, 1_048_840, "f32"),      # 16,392 partials, ragged last segment: 9 blocks, tails only
    (8, 262_144, "bf16"),       # 8,192 partials: 4 blocks of 2,048, four terms per thread
])
def test_finalize_equals_exact_sum_of_its_partials(N, C, gdt):
    P = N * C
    w = I.TINY.with_(N=N, P=P, gdtype=gdt, grad=I.Dist(I.NORMAL, 1.0), grad_seed=17)
    G = torch.empty(N * P, dtype=torch.bfloat16 if gdt == "bf16" else torch.float32, device=DEV)
    _wide(w, G)
    ws, norm, n = _norm(G, N, P)
    parts = _partials(ws, n)
    assert np.all(np.isfinite(parts)) and np.all(parts >= 0)
    exact = math.fsum(parts.tolist())
    got = _sumsq(ws)
    # Sum2 per chain of k terms: within gamma(k-1)^2 of the chain's sum; the
    # fp64 tree and second stage add a few units of 2^-53
    assert abs(got - exact) <= 1e-12 * exact, (got, exact)
    if n <= 20_000:        # the documented order, bit for bit (host emulation)
        assert np.float64(got).tobytes() == np.float64(_emulated_sumsq(parts)).tobytes()
    # against the fp64 sum of squares of the values themselves: the segments'
    # fp32 trees are the only other rounding (bound 8 * 2^-24 relative)
    ref = _owner_sumsq(G, N, P)
    assert abs(norm - math.sqrt(ref)) <= 1e-6 * math.sqrt(ref), (norm, math.sqrt(ref))
    assert _dpz().ws_status(ws) == 0


def _mid_arena(seed=5):
    N, C = 4, 1_048_840
    P = N * C
    w = I.TINY.with_(N=N, P=P, gdtype="f32", grad=I.Dist(I.NORMAL, 1.0), grad_seed=seed)
    G = torch.empty(N * P, dtype=torch.float32, device=DEV)
    I.fill_grads_device(w, G)
    return N, C, P, G


def test_overflowing_chain_is_added_in_fp64():
    """Owner values in [0.9e18, 1e18]: every segment's fp32 sum of squares
    (2.1e38 to 2.6e38) is finite, the fp32 sum of two of them is not; every
    chain is added again in fp64 and the norm is finite and correct."""
    N, C, P, G = _mid_arena()
    g = G.view(N, P)
    for c in range(N):
        g[c, c * C:(c + 1) * C].uniform_(0.9e18, 1e18)
    ws, norm, n = _norm(G, N, P)
    parts = _partials(ws, n)
    assert np.all(np.isfinite(parts)) and parts.max() > 1e38
    exact = math.fsum(parts.tolist())
    assert exact > 3.5e38                              # beyond fp32
    assert abs(_sumsq(ws) - exact) <= 1e-12 * exact
    assert np.float64(_sumsq(ws)).tobytes() == np.float64(_emulated_sumsq(parts)).tobytes()
    ref = math.sqrt(_owner_sumsq(G, N, P))
    assert math.isfinite(norm) and abs(norm - ref) <= 1e-6 * ref, (norm, ref)
    assert _dpz().ws_status(ws) == 0


def test_subnormal_partials_are_added_in_fp64():
    """A chunk of values near 1e-21: its segments' sums of squares are fp32
    subnormals, whose chains are added in fp64; the rest take the fp32 path."""
    N, C, P, G = _mid_arena(6)
    g = G.view(N, P)
    g[1, C:2 * C].mul_(1e-21)
    ws, norm, n = _norm(G, N, P)
    parts = _partials(ws, n)
    segs = n // N
    tiny = parts[segs:2 * segs]
    assert np.all(tiny < np.float32(1.1754944e-38)) and np.any(tiny > 0)   # subnormal in fp32
    exact = math.fsum(parts.tolist())
    assert abs(_sumsq(ws) - exact) <= 1e-12 * exact
    assert np.float64(_sumsq(ws)).tobytes() == np.float64(_emulated_sumsq(parts)).tobytes()
    ref = math.sqrt(_owner_sumsq(G, N, P))
    assert abs(norm - ref) <= 1e-6 * ref
    assert _dpz().ws_status(ws) == 0


@pytest.mark.parametrize("bad", [float("nan"), float("inf")])
def test_nonfinite_value_in_a_long_chain(bad):
    N, C, P, G = _mid_arena(7)
    G.view(N, P)[2, 2 * C + 777] = bad
    ws, norm, n = _norm(G, N, P)
    if math.isnan(bad):
        assert math.isnan(norm) and math.isnan(_sumsq(ws))
    else:
        assert norm == math.inf and _sumsq(ws) == math.inf
    assert _dpz().ws_status(ws) == 0       # a non-finite norm is data, not a skipped tile


@pytest.mark.parametrize("marker,status", [(-1.0, 1), (-2.0, 3)])
def test_marker_partial_in_a_long_chain(marker, status):
    """A skipped tile's marker written into one partial (host-side, between
    calls): the finalisation reports it in the status word and a NaN norm;
    with the partial restored it gives the first result's bits again."""
    dpz = _dpz()
    N, C, P, G = _mid_arena(8)
    ws, norm0, n = _norm(G, N, P)
    k = n // 2 + 3
    pv = ws[PARTIALS_AT:PARTIALS_AT + 8 * n].view(torch.float64)
    keep = pv[k].item()
    pv[k] = marker
    nrm = torch.zeros(1, device=DEV)
    dpz.dp_grad_norm_finalize(ws, P, N, nrm)
    torch.cuda.synchronize()
    assert math.isnan(nrm.item()) and math.isnan(_sumsq(ws))
    assert dpz.ws_status(ws) == status
    pv[k] = keep
    dpz.dp_grad_norm_finalize(ws, P, N, nrm)
    torch.cuda.synchronize()
    assert np.float32(nrm.item()).tobytes() == np.float32(norm0).tobytes()
    assert dpz.ws_status(ws) == 0
