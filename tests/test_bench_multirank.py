"""bench.py's multi-rank host logic with two gloo ranks on the CPU."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = torch.multiprocessing


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 5.0 - rank, 2.0 * rank, 0.5]
        got = bench.max_over_ranks(mine)
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert res[0] == res[1] == [2.0, 5.0, 2.0, 0.5]


def test_single_process_is_identity_and_value_scales_with_ranks():
    import bench
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    one = bench.aggregate_value(68.72e9, 0.1, 1)
    two = bench.aggregate_value(68.72e9, 0.1, 2)
    assert abs(one - 687.2) < 1e-6 and abs(two - 2 * one) < 1e-9
