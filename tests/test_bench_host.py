"""bench.py's host logic without a GPU: the algorithmic byte counts, the
max-over-ranks timing on a world-size-2 gloo group, and the reference arm's
JSON line."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

import bench
import inputs as I
from conftest import ROOT


def test_step_bytes_match_the_minimal_traffic_formula():
    # N*P*e_g + 24*P + N*P*e_w: 40P for N = 4 bf16, 56P for N = 8 bf16
    assert bench.step_bytes(I.GPT2_1P5B) == 40 * 1_557_611_200 == 62_304_448_000
    assert bench.step_bytes(I.GPT2_124M) == 56 * 124_439_808
    assert bench.step_bytes(I.TINY) == 4 * 4096 * 4 + 24 * 4096 + 4 * 4096 * 2 == 196_608
    assert bench.step_bytes(I.ALLREDUCE_7B) == 2 * 4 * 7_000_000_000 * 2
    # with clipping, the three kernels move 44P for the 1.5B workload
    w = I.GPT2_1P5B
    k = sum(bench.kernel_bytes(n, w) for n in ("dpz_rs_avg_sumsq", "dpz_adamw_bcast"))
    assert k == 44 * w.P


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    m = bench.max_over_ranks(1.5 + rank, world)
    bench.barrier(world)
    q.put((rank, m))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 2.5, 1: 2.5}


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", I.TINY.name, "--steps", "2", "--warmup", "0",
                          "--ref-seconds", "0.2"], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["metric"] == bench.METRIC


def test_reference_arm_nonzero_rank_does_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", I.TINY.name, "--steps", "1", "--warmup", "0"],
                         capture_output=True, text=True, timeout=120, env=env)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_cpu_baselines_single_and_threaded():
    """The oracle timed on one thread and on several disjoint windows at once."""
    one = bench.time_oracle(I.GPT2_124M, 0.2)
    many = bench.time_oracle_threads(I.GPT2_124M, 0.2, 2)
    for r, cores in ((one, 1), (many, 2)):
        assert r["kind"] == "oracle" and r["unit"] == bench.UNIT and r["cores"] == cores
        assert r["value"] > 0 and "windows" in r["sample"]


def test_l2_note_says_which_workloads_stream_from_hbm():
    assert bench.l2_note(I.GPT2_1P5B).startswith("inputs larger than L2")
    assert bench.l2_note(I.ALLREDUCE_7B).startswith("inputs larger than L2")
    assert bench.touched_bytes(I.ALLREDUCE_7B) == 4 * 7_000_000_000 * 2
    assert "L2 reuse" in bench.l2_note(I.TINY)
    assert "L2 reuse" in bench.l2_note(I.allreduce_sweep(16 << 20, 4))     # 64 MiB arena
    assert bench.l2_note(I.allreduce_sweep(1 << 30, 2)).startswith("inputs larger than L2")


def test_kernel_traffic_follows_its_own_sources(tmp_path, monkeypatch):
    """A kernel's ncu traffic is used while its translation unit hashes as it
    did at capture: a code change in it drops the figure, a comment-only
    change or a change to another kernel's file does not."""
    import shutil
    src = tmp_path / "csrc"
    shutil.copytree(bench.CSRC, src)
    monkeypatch.setattr(bench, "CSRC", str(src))
    w = I.GPT2_1P5B
    before = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_UNITS}
    with open(src / "adamw.cu", "a") as f:          # in no unit of the table
        f.write("\nstatic int unrelated_change = 1;\n")
    with open(src / "reduce.cu", "a") as f:         # comment only
        f.write("\n// a remark\n/* and another */\n")
    assert {k: bench.kernel_source_hash(k) for k in bench.KERNEL_UNITS} == before
    with open(src / "reduce.cu", "a") as f:         # code: only the reduce unit changes
        f.write("\nstatic int changed = 2;\n")
    after = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_UNITS}
    assert after["dpz_rs_avg_sumsq"] != before["dpz_rs_avg_sumsq"]
    assert after["dpz_adamw_bcast"] == before["dpz_adamw_bcast"]
    assert after["dpz_zero1_fused_sumsq"] == before["dpz_zero1_fused_sumsq"]
    # every kernel of the committed table has a unit and a recorded hash
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        table = json.load(f)
    assert set(table["kernels"]) == set(bench.KERNEL_UNITS)
    assert all(len(k["source_hash"]) == 16 for k in table["kernels"].values())


def test_clock_record_rejection_rule():
    """A slowdown or a clock stuck well below its maximum with no reason makes
    the timed region invalid (bench.py then takes it again once); the power
    cap alone does not."""
    import bench
    full = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 9}
    assert not bench.clocks_rejected(None)
    assert not bench.clocks_rejected(full)
    assert not bench.clocks_rejected(dict(full, sm_mhz=1900.0, reasons=["sw_power_cap"]))
    assert not bench.clocks_rejected(dict(full, sm_mhz=1500.0, reasons=["sw_power_cap"]))
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected(dict(full, reasons=[r]))
    assert bench.clocks_rejected(dict(full, sm_mhz=1200.0))          # a leftover clock lock
    assert not bench.clocks_rejected(dict(full, sm_mhz=1950.0))
