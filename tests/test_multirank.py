"""The multi-rank host logic of bench.py, on CPU processes with the gloo backend (world size 2).

bench.py runs one independent replica of the workload per rank (the path has no exchange step);
what ranks share is the timing: every rank must end with the slowest rank's time, and the
whole-job rate counts the units of every rank.  The reference arm runs on rank 0 only.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank                       # rank 1 is the slow one
        got = bench.max_over_ranks(mine, dist, torch.device("cpu"))
        rate = bench.whole_job_rate(world, 1000.0, got)
        out[rank] = (got, rate)
    finally:
        dist.destroy_process_group()


def test_timing_is_the_max_over_ranks_and_rate_counts_every_rank():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] == res[1][1] == pytest.approx(2 * 1000.0 / 0.015)


def test_single_process_needs_no_collective():
    import bench
    assert bench.max_over_ranks(3.5, None, torch.device("cpu")) == 3.5
    assert bench.whole_job_rate(1, 500.0, 2.0) == pytest.approx(250000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    from selective_state_space_gb300 import workloads
    monkeypatch.setenv("RANK", "1")

    class Args:
        warmup, steps, ref_step_s = 3, 1, 1.0

    assert bench.run_reference(Args(), workloads.WORKLOADS[0]) is None
    assert capsys.readouterr().out == ""
