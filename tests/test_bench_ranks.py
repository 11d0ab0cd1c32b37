"""The bench's multi-rank host logic on CPU: two gloo ranks (replicas only - the path has
no data exchange), the max-over-ranks step time, the whole-job GB/s, and the reference
arm's other ranks leaving without work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        # each rank's own timed region; the slowest one sets the step
        got = bench.ranks_max(dist, 10.0 * (rank + 1))
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        assert dict(out) == {0: 20.0, 1: 20.0}


def test_whole_job_value_sums_the_ranks():
    # 2 ranks x 2.477 GB each in 0.365 ms: twice one rank's rate
    one = bench.job_gbps(1, 2_477_260_800, 0.365)
    assert bench.job_gbps(2, 2_477_260_800, 0.365) == pytest.approx(2 * one)
    assert one == pytest.approx(2_477_260_800 / 0.365e-3 / 1e9)
    assert bench.ranks_max(None, 3.5) == 3.5


def test_reference_arm_other_ranks_do_nothing(capsys):
    # rank 1 of 2 returns before reading its arguments: no work, no output
    assert bench.run_reference(None, 2, 1) is None
    assert capsys.readouterr().out == ""


def test_replica_seeds_differ_per_rank():
    from datagen import workloads as W
    seeds = {W.decode_seed(layer + 1000 * rank, proj) for rank in (0, 1) for layer in (0, 34) for proj in range(7)}
    assert len(seeds) == 2 * 2 * 7
