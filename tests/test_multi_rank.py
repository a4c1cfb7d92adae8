"""The benchmark's multi-rank (replica) aggregation on CPU with gloo,
world size 2: the step time is the slowest rank's and the value counts the
bytes of every rank.  The GEMV path does not shard, so ranks are replicas."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [1.5, 2.25][rank]
    slowest = bench.slowest_rank_ms(ms, world)
    out[rank] = (slowest, bench.job_value(1_000_000, slowest, world))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(2, _free_port(), out), nprocs=2, start_method="spawn", join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.25
    assert res[0][1] == pytest.approx(2 * 1_000_000 / 2.25e-3 / 1e9)


def test_single_rank_is_identity():
    import bench
    assert bench.slowest_rank_ms(3.0, 1) == 3.0
    assert bench.job_value(2_000_000, 1.0, 1) == pytest.approx(2.0)
