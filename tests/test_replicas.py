"""The multi-GPU form of the bench is replicas only (the decode step has no
cross-GPU exchange): each rank decodes its own sequence and the job's time is
the slowest rank's.  These tests run the host side of that path as two gloo
ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    ws, r, local = bench.dist_env()
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # rank r took 1 + r seconds for 10 steps
        t = bench.max_over_ranks(1.0 + rank, dist, torch.device("cpu"))
        dist.barrier()
        out[rank] = (ws, r, local, t, bench.job_throughput(ws, 10, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:  # no fork of this (threaded) process
        out = mgr.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        ws, r, local, t, value = res[rank]
        assert (ws, r, local) == (2, rank, rank)
        assert t == 2.0  # every rank sees the slowest rank's time
        assert value == pytest.approx(10.0)  # 2 replicas x 10 steps / 2 s


def test_single_process_needs_no_collective():
    assert bench.max_over_ranks(1.5, None, torch.device("cpu")) == 1.5
    assert bench.job_throughput(1, 128, 2.0) == 64.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    """Under torchrun the oracle arm's other ranks exit 0 at once, printing nothing."""
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.run_reference(bench.parse_args(["--impl", "reference", "--gpus", "2", "--workload", "tiny"])) == 0
    assert capsys.readouterr().out == ""
