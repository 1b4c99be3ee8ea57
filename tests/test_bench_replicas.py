"""The multi-GPU path of bench.py is N independent replicas (decode rows are independent, so
the step needs no exchange): the reported time is the slowest rank's, the units are every
rank's.  Checked with two gloo processes on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, units = bench.replica_aggregate(10.0 + 5.0 * rank, 32 * (rank + 1), world)
    out[rank] = (ms, units)
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replica_aggregate_takes_the_slowest_rank_and_all_units(world):
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        ms, units = out[r]
        assert ms == 10.0 + 5.0 * (world - 1)
        assert units == sum(32 * (k + 1) for k in range(world))


def test_single_process_passes_through():
    import bench
    assert bench.replica_aggregate(3.5, 7, 1) == (3.5, 7)
