"""The N > 1 bench path on CPU: two gloo ranks (one process each, as under
torchrun) check the replica timing rule (the slowest rank's time, units of all
ranks) and that the reference arm runs on rank 0 only."""
import argparse
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench._dist() == (rank, world, rank)
        # rank r took 10 + 5 r ms for 320 tokens
        value, ms = bench._whole_job_rate(320, 10.0 + 5.0 * rank, world, "cpu")
        # rank 1 of the reference arm returns at once, printing nothing
        a = argparse.Namespace(workload="tiny_fp32", a_max=None, warmup=0, steps=1)
        ran = bench.run_reference(a) if rank == 1 else None
        out[rank] = (value, ms, ran)
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    for rank in range(world):
        value, ms, ran = res[rank]
        assert ms == 15.0                        # max over ranks
        assert value == pytest.approx(320 * 2 / 0.015)
        assert ran is None


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    value, ms = bench._whole_job_rate(64, 8.0, 1, "cpu")
    assert ms == 8.0 and value == pytest.approx(8000.0)
