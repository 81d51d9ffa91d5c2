"""The multi-GPU path is replicas only: each rank serves its own step, the
job's time is the slowest rank's, and no data crosses ranks.  The host logic
of that reduction runs here on CPU with two gloo ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [1.5, 2.25][rank]
    slowest = bench.max_over_ranks(ms)
    out[rank] = (slowest, bench.replica_throughput(256, slowest, world), bench.dist_info())
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        slowest, value, info = res[rank]
        assert slowest == 2.25
        assert value == pytest.approx(2 * 256 / 2.25e-3)
        assert info[0] == rank and info[1] == 2


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.0) == 3.0
    assert bench.replica_throughput(256, 2.0, 1) == pytest.approx(128000.0)
