"""The layouts' memory per simulated rank against the ZeRO model-state table
of "Lab 09 — Parallelism, simulated", §4."""
import pytest

from gradient_reduction_zero_gb300 import memory as Mem


@pytest.fixture(scope="module")
def table(golden):
    return [(float(p), int(n), int(s), float(gb)) for p, n, s, gb in golden("zero_memory.txt")]


def test_model_reproduces_the_lab_table(table):
    for params, N, stage, gb in table:
        got = Mem.zero_model_state_bytes(params, N, stage) / 1e9
        # the table rounds to 3 significant digits (31.40625 -> 31.4, 16.64 -> 16.6)
        assert abs(got - gb) <= 0.005 * gb, (params, N, stage, got, gb)


@pytest.mark.parametrize("params,N", [(7.5e9, 64), (7e9, 8), (1_557_611_200, 4), (124_439_808, 8)])
def test_layouts_hold_what_the_stages_allow(params, N):
    P = int(params) // (8 * N) * 8 * N
    z1 = Mem.rank_buffers(P, N, "zero1")
    z2 = Mem.rank_buffers(P, N, "zero2", bucket=1 << 20)
    assert Mem.model_state_bytes(z1) == pytest.approx(Mem.zero_model_state_bytes(P, N, 1), rel=0,
                                                      abs=1)
    assert Mem.model_state_bytes(z2) == pytest.approx(Mem.zero_model_state_bytes(P, N, 2), rel=0,
                                                      abs=1)
    # ZeRO-2 drops the full gradient replica: 2P (1 - 1/N) bytes less per rank
    assert Mem.model_state_bytes(z1) - Mem.model_state_bytes(z2) == 2 * P - 2 * (P // N)


def test_gpt2_1p5b_arena_at_n4():
    """The benchmark's arena: 43.6 GB for four simulated ranks under ZeRO-1."""
    P, N = 1_557_611_200, 4
    per_rank = Mem.model_state_bytes(Mem.rank_buffers(P, N, "zero1"))
    assert abs(N * per_rank / 1e9 - 43.6) < 0.05
