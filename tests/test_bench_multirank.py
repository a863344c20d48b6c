"""The N>1 host path of bench.py on CPU: two gloo ranks with different
timings agree on the max, and the whole-job value counts every rank's work
over the slowest rank's time (independent replicas, weak scaling)."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mx = bench.max_over_ranks([10.0 + rank, 5.0 - rank, 3.0 * (rank + 1)], dist)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, mx))


def test_two_gloo_ranks_take_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[0] == out[1] == [11.0, 5.0, 6.0]


def test_aggregate_value_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_value(2 * 10**12, 1, 2.0) == pytest.approx(1000.0)
    assert bench.aggregate_value(2 * 10**12, 4, 2.0) == pytest.approx(4000.0)
