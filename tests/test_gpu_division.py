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

