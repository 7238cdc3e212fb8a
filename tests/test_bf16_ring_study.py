"""The rounding study of "13.5 Multi-GPU from First Principles", Exercise 8,
on synthetic shard gradients.

Each of k shards has gradient g_r = mu + eta_r with a common component mu
and a shard-specific one eta_r, both N(0, 1) per element, so two shards'
gradients differ by about as much as they agree (the pages use LeNet
gradients on Fashion-MNIST shards; no dataset is used here).  Two bf16 rings
average them:

  per-hop:  inputs rounded to bf16, partial sum rounded to bf16 after every
            hop (the default ring, DPZ_BF16);
  acc32:    inputs rounded to bf16 once, partial sums in fp32, the average
            rounded to bf16 once (DPZ_BF16_ACC32).

Both are compared with the exact mean of the fp32 gradients (fp64).  Run
with -s to print the table.

The per-hop ring rounds a partial sum that grows with the hop count. Its
error compounds like a random walk over k roundings, each of relative size
about 2^-9 of the current partial sum. The relative error therefore grows
with k, roughly as sqrt(k).

The fp32-accumulating ring loses almost nothing in the sum. Its error is
the input roundings, which average down, plus the one final rounding, so it
stays near the bf16 rounding floor whatever k is.

Both errors are far below the difference between two shards' gradients,
which is of order 1.  So the rounding does not matter for SGD; the pages'
part (b) asks for exactly this comparison.
"""
import numpy as np
import pytest

import oracle as O

KS = (2, 8, 64)


def shard_grads(k, P, seed=0):
    rng = np.random.default_rng(seed)
    mu = rng.standard_normal(P)
    return np.stack([(mu + rng.standard_normal(P)).astype(np.float32) for _ in range(k)])


def rel_err(avg_bf16_owner, ref):
    got = O.bf16_to_f32(avg_bf16_owner).astype(np.float64)
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def study(P=1 << 16):
    rows = []
    for k in KS:
        g = shard_grads(k, P, seed=k)
        ref = g.astype(np.float64).mean(axis=0)
        C = P // k
        res = {}
        for mode, acc32 in (("per-hop", False), ("acc32", True)):
            a = O.f32_to_bf16(g)
            O.reduce_scatter_avg(a, acc32=acc32)
            owner = np.concatenate([a[c, c * C:(c + 1) * C] for c in range(k)])
            res[mode] = rel_err(owner, ref)
        spread = float(np.linalg.norm(g[0].astype(np.float64) - g[1]) / np.linalg.norm(g[0]))
        rows.append((k, res["per-hop"], res["acc32"], spread))
    return rows


def test_bf16_ring_rounding_study():
    rows = study()
    print("\n  k   per-hop rel. err   acc32 rel. err   shard-to-shard rel. diff")
    for k, a, b, d in rows:
        print(f"{k:3d}   {a:14.3e}   {b:14.3e}   {d:10.3f}")
    err = {k: (a, b) for k, a, b, _ in rows}
    # per-hop rounding error grows with k; fp32 accumulation stays at the floor
    assert err[64][0] > 3.0 * err[2][0]
    assert err[64][1] < 1.5 * err[2][1]
    for k in (8, 64):
        assert err[k][0] > err[k][1]
    # the floor is one bf16 rounding: relative error near 2^-9 / sqrt(3)
    for k in KS:
        assert 2.0 ** -12 < err[k][1] < 2.0 ** -8
    # rounding is tiny next to the gradient differences between shards
    for _, a, b, d in rows:
        assert max(a, b) < 1e-2 * d


@pytest.mark.parametrize("k", KS)
def test_study_inputs_are_exact_for_the_ring(k):
    """The study's inputs satisfy the ring's layout (P a multiple of 8k)."""
    assert (1 << 16) % (8 * k) == 0
