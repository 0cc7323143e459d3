"""The multi-rank host logic of bench.py, run as two gloo ranks on the CPU:
each rank gets a shard of its own (same geometry, different requests), the
step time is the maximum over ranks, and the whole-job value counts every
rank's units. No GPU and no collective on the data path."""
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench
    import synth

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        base = synth.tiny_05b()
        spec = bench.rank_spec(base, rank)
        # same geometry and sizes on every rank
        geo = torch.tensor([spec.L, spec.H, spec.D, spec.bs, spec.R, spec.total_blocks, spec.num_pages],
                           dtype=torch.int64)
        geos = [torch.zeros_like(geo) for _ in range(world)]
        dist.all_gather(geos, geo)
        # its own requests: the page tables and random streams differ between ranks
        fp = torch.tensor([spec.key & 0x7FFFFFFFFFFFFFFF, int(np.asarray(spec.pages).sum())], dtype=torch.int64)
        fps = [torch.zeros_like(fp) for _ in range(world)]
        dist.all_gather(fps, fp)
        # the slowest rank's time is the job's time
        local_ms = 10.0 + 5.0 * rank
        got = bench.max_over_ranks(local_ms)
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(" ".join(str(int(x)) for g in geos for x in g) + "\n")
            f.write(" ".join(str(int(x)) for g in fps for x in g) + "\n")
            f.write(repr(got) + "\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp

    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    lines = [open(tmp_path / f"rank{r}.txt").read().split("\n") for r in range(world)]
    for r in range(world):
        geo = [int(x) for x in lines[r][0].split()]
        assert geo[:7] == geo[7:], "ranks must run the same geometry"
        fps = [int(x) for x in lines[r][1].split()]
        assert fps[0] != fps[2], "ranks must draw different requests"
        assert float(lines[r][2]) == 15.0, "max over ranks"


def test_rank_zero_keeps_the_workload_seed():
    sys.path.insert(0, ROOT)
    import bench
    import synth

    base = synth.tiny_05b()
    assert bench.rank_spec(base, 0) is base
    other = bench.rank_spec(base, 3)
    assert other.seed != base.seed and other.total_blocks == base.total_blocks


def test_weak_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench

    # 2 ranks x 4 GB per step x 10 steps in 20 ms (slowest rank) = 4000 GB/s
    assert bench.weak_value(4e9, 10, 2, 20.0) / 1e9 == pytest.approx(4000.0)
    assert bench.max_over_ranks(3.5) == 3.5  # no process group: the value itself


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--workload", "tiny"], env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


def test_clock_summary_uses_the_timed_window():
    sys.path.insert(0, ROOT)
    import bench

    row = lambda mhz, cap="Not Active": f"{mhz}, 2070, Not Active, Not Active, Not Active, {cap}"  # noqa: E731
    lines = [(0.0, row(1000)), (1.0, row(1900)), (1.1, row(2000, "Active")), (1.2, row(2070)), (2.0, row(900))]
    s = bench.summarize_clocks(lines, 0.9, 1.25)
    assert s["samples"] == 3 and s["sm_mhz"] == 2000 and s["reasons"] == ["sw_power_cap"] and s["in_window"]
    s = bench.summarize_clocks(lines, 1.3, 1.4)  # window shorter than the period: next sample, flagged
    assert s["samples"] == 1 and s["sm_mhz"] == 900 and not s["in_window"]
    assert bench.summarize_clocks([], 0, 1)["samples"] == 0


def test_pool_profile_is_of_the_current_sources():
    """The bench reports the headline pool's DRAM traffic from the committed
    ncu summary only while the kernels' sources hash to the profiled ones: a
    change to those sources needs the counters taken again."""
    sys.path.insert(0, ROOT)
    import bench

    traffic = bench.profiled_traffic(bench.DEFAULT_WORKLOAD)
    assert traffic is not None, "the weighted pool's ncu summary was taken on other kernel sources"
    # one weighted pool call reads the 120.26 GB of K once, plus its 1/64-size slice sums
    assert 1.20e11 < traffic < 1.30e11
