"""The multi-rank host logic of bench.py on CPU: two gloo ranks (127.0.0.1).

Each GPU of a multi-GPU run is an independent replica; the only exchange is
the max over ranks of the timed region, and the reported value is the
whole-job throughput.  The reference arm prints from rank 0 only.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slower one
        got = bench.max_over_ranks(torch, dist, ms, torch.device("cpu"), world)
        dist.barrier()
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(torch, None, 12.5, torch.device("cpu"), 1) == 12.5


def test_job_value_is_whole_job_throughput():
    # 2 replicas x 1 GB per step in 1 ms -> 2000 GB/s
    assert bench.job_value(2, 1e9, 1.0) == pytest.approx(2000.0)
    assert bench.job_value(1, 711741488.0, 0.3662) == pytest.approx(1943.6, rel=1e-3)


def test_reference_arm_prints_on_rank0_only(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 1, 3
    bench.run_reference(Args())
    assert capsys.readouterr().out == ""


def test_replica_command_starts_one_rank_per_gpu():
    """--gpus N without a launcher re-runs the benchmark as N ranks on 127.0.0.1."""
    cmd = bench.replica_command(["--gpus", "4", "--steps", "5"], 4, 29511)
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"]
    assert "--nproc-per-node=4" in cmd
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[cmd.index("--master-port") + 1] == "29511"
    assert cmd[-4:] == ["--gpus", "4", "--steps", "5"] and cmd[-5].endswith("bench.py")
