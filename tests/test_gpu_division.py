"""The average divides the reduced sum by N ("Lab 09 — Parallelism, simulated",
§2: sum, then divide by N).  For N not a power of two the kernels divide with
Markstein's correction of a reciprocal product; this checks,
through the library's own division routine, that the quotient equals the IEEE
round-to-nearest quotient for every one of the 2^32 float bit patterns and
every N the library accepts (1 to 64)."""
import pytest
import torch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import gradient_reduction_zero_gb300.dpz as dpz
    from gpu_util import DEV

NS = list(range(1, 65))


def test_average_division_is_correctly_rounded_for_every_float():
    counters = torch.full((len(NS), 2), -1, dtype=torch.int64, device=DEV)
    for i, N in enumerate(NS):
        dpz.selftest_average_division(N, counters[i, :1])
    torch.cuda.synchronize()
    bad = {N: int(c) for N, c in zip(NS, counters[:, 0].tolist()) if c != 0}
    assert bad == {}, bad



@pytest.mark.parametrize("N", [3, 7])
def test_acc32_reduce_on_sums_next_to_bf16_ties(N):
    """End to end through the fp32-accumulating reduce-scatter: sums whose
    quotient by N sits next to a bf16 tie, where a reciprocal product would
    change the bf16 average, each split into three exact bf16 parts on the
    first ranks of chunk 0's ring order.  The averages equal the oracle's bit
    for bit."""
    import numpy as np
    import oracle as O
    from gpu_util import down, up
    rng = np.random.default_rng(100 + N)
    bits = rng.integers(0x3F800000, 0x40000000, 2_000_000, dtype=np.uint32)   # [1, 2)
    s = bits.view(np.float32)

    def bf16_bits(x):
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
            torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    q_ieee = (s.astype(np.float64) / N).astype(np.float32)
    q_recip = (s * (np.float32(1) / np.float32(N))).astype(np.float32)
    sums = s[np.nonzero(bf16_bits(q_ieee) != bf16_bits(q_recip))[0][:8]]
    assert len(sums) >= 2
    C = 1024
    x = np.zeros((N, N * C), dtype=np.float32)
    for e, a in enumerate(sums):
        hi = (np.array([a]).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)[0]
        rem = np.float32(a - hi)
        mid = (np.array([rem]).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)[0]
        x[1, e], x[2, e], x[3 % N, e] = hi, mid, np.float32(rem - mid)
    xb = O.f32_to_bf16(x)
    G = up(xb)
    dpz.dp_reduce_scatter_avg(G, N, acc32=True)
    torch.cuda.synchronize()
    want = xb.copy()
    O.reduce_scatter_avg(want, acc32=True)
    got = down(G).reshape(N, N * C)
    assert np.array_equal(got[0, :C], want[0, :C])
