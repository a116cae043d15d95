"""The N > 1 bench path on CPU: independent replicas, max-over-ranks timing over gloo (world 2)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as tdist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed = bench.reduce_max(1.0 + rank)          # rank 1 is the slow one
    out[rank] = (elapsed, bench.replica_throughput(world, 1e9, 10, elapsed))
    tdist.barrier()
    tdist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        elapsed, value = out[r]
        assert elapsed == 2.0                       # every rank sees the slowest rank's time
        assert value == pytest.approx(world * 1e9 * 10 / 2.0 / 1e9)


def test_single_process_identity():
    import bench
    assert bench.reduce_max(3.5) == 3.5
    assert bench.replica_throughput(1, 2e9, 4, 2.0) == pytest.approx(4.0)
