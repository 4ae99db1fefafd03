"""The replica path of bench.py across two ranks (gloo, CPU): the whole-job
throughput is every rank's tokens over the slowest rank's time."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    secs, tokens = bench.aggregate(1.0 + rank, 100 * (rank + 1), dist, "cpu")
    out[rank] = (secs, tokens)
    dist.destroy_process_group()


def test_two_replicas_aggregate():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    # slowest rank: 2 s; tokens: 100 + 200
    assert res[0] == (2.0, 300) and res[1] == (2.0, 300)


def test_single_process_aggregate_is_identity():
    import bench
    assert bench.aggregate(3.5, 42) == (3.5, 42)
