"""The bench's multi-rank host logic on CPU ranks (gloo, world size 2): the
job time is the maximum over ranks, and the reference arm runs on rank 0
only. Every rank runs an independent replica (the path has no exchange)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r reports (r + 1, 10 - r): the maxima are (world, 10)
        out[rank] = bench.reduce_max((rank + 1.0, 10.0 - rank), world, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        assert out[0] == (2.0, 10.0) and out[1] == (2.0, 10.0)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import argparse

    import bench
    args = argparse.Namespace(gpus=2, steps=1, warmup=0)
    bench.run_reference(args, rank=1, world=2)  # returns at once, prints nothing
    assert capsys.readouterr().out == ""


def test_single_rank_reduce_is_identity():
    import bench
    assert bench.reduce_max((1.5, 2.5), 1, "cpu") == (1.5, 2.5)
