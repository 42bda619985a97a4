"""Host logic of the multi-process bench on CPU: world size 2 over gloo.

The decode layer has no exchange step, so N GPUs run N independent replicas;
the job's throughput is the units of all ranks over the slowest rank's time.
These tests run that aggregation (and the barrier) in two processes."""
import os
import socket

import pytest


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
    try:
        import bench
        bench.barrier(world)
        units = [1000.0, 3000.0][rank]
        secs = [1.0, 2.0][rank]
        q.put((rank, bench.reduce_max(secs, world), bench.reduce_sum(units, world),
               bench.replica_throughput(units, secs, world)))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_replica_aggregation_world2():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, tmax, usum, thr in res:
        assert tmax == 2.0 and usum == 4000.0
        assert thr == pytest.approx(2000.0)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.reduce_sum(7.0, 1) == 7.0
    assert bench.replica_throughput(10.0, 2.0, 1) == 5.0
