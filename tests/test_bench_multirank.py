"""bench.py's multi-rank logic on CPU (gloo, world size 2): each rank runs its
own batch (weak scaling, no collective on the data path); the whole-job
value sums the ranks' units and divides by the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    units = 1000.0 * (rank + 1)          # different batches per rank
    seconds = 0.5 + 0.25 * rank          # rank 1 is slower
    u, t = bench.aggregate(units, seconds, dist)
    q.put((rank, u, t))
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_sums_units_and_takes_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, u, t in results:
        assert u == pytest.approx(3000.0)
        assert t == pytest.approx(0.75)


def test_aggregate_single_process_is_identity():
    import bench
    assert bench.aggregate(12.0, 3.0, None) == (12.0, 3.0)
