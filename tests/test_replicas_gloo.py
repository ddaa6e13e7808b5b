"""The multi-GPU mode is N independent replicas: bench.py's ranks meet at a
barrier, take the slowest rank's time and report the whole-job rate.  These
tests run that host-side logic as two gloo ranks on the CPU (no GPU needed)."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

from conftest import ROOT

sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup()
    try:
        assert (r, w, local) == (rank, world, rank)
        bench.barrier(w)
        ms = 10.0 * (rank + 1)                     # rank 1 is the slower one
        ms_max, value = bench.job_throughput(ms, 1000, w)
        line = bench.run_reference(None, r, w) if r != 0 else "rank0"
        q.put((rank, ms_max, value, line))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=100) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for rank, ms_max, value, line in got:
        assert ms_max == 20.0                      # every rank sees the max over ranks
        assert value == pytest.approx(2 * 1000 / 0.020)   # both ranks' steps over the slowest time
    assert got[1][3] is None                       # only rank 0 runs the reference arm


def test_single_process_needs_no_process_group():
    import bench
    assert bench.job_throughput(5.0, 100, 1) == (5.0, 100 / 0.005)
    bench.barrier(1)   # no-op without a process group


@pytest.mark.timeout(300)
def test_reference_arm_times_exactly_the_requested_rounds():
    """bench.py --impl reference on rank 0: W untimed and exactly K timed rounds of one
    oracle C2 step per usable core; the line reports K and W and a positive rate."""
    import argparse
    import bench
    line = bench.run_reference(argparse.Namespace(steps=2, warmup=1), 0, 1)
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    cores = line["cpu_baseline"]["cores"]
    assert cores == bench.cpu_cores() >= 1
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
    assert f"{2 * cores} steps" in line["cpu_baseline"]["sample"]
    assert line["ms_per_step"] > 0 and line["dtype"] == "f64"
