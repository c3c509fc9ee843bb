"""The N > 1 path of bench.py on CPU: independent replicas, one per rank,
with no collective on the data path; the only exchange is the slowest rank's
time, taken after the timed region (two gloo ranks on 127.0.0.1)."""
import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(times[rank], dist, "cpu")
        value = bench.whole_job_rate(world, 1, 128, slowest)
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [0.75, 1.25]
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, times, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == 1.25
        assert value == pytest.approx(2 * 128 / 1.25)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(0.5, None, "cpu") == 0.5
    assert bench.whole_job_rate(1, 8, 64, 2.0) == 256.0


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import argparse
    import synth
    args = argparse.Namespace(steps=1, warmup=3)
    assert bench.reference_arm(args, synth.workload("tiny"), rank=1, world=2) == 0
    assert capsys.readouterr().out == ""
