"""The benchmark's replica bookkeeping across processes (gloo, world size 2,
CPU): barriers line up, the reported time is the slowest rank's, and the
work is summed over ranks."""
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

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rep = bench.Replicas(dist, world)
    rep.barrier()
    ms = rep.max(10.0 + 5.0 * rank)          # rank 1 is the slow one
    units = rep.sum(1000.0 * (rank + 1))     # ranks did 1000 and 2000 units
    rate = bench.throughput(units, ms)
    rep.barrier()
    dist.destroy_process_group()
    q.put((rank, ms, units, rate))


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, units, rate in res:
        assert ms == 15.0 and units == 3000.0
        assert rate == pytest.approx(3000.0 / 0.015)


def test_single_process_is_identity():
    import bench
    rep = bench.Replicas(None, 1)
    rep.barrier()
    assert rep.max(3.5) == 3.5 and rep.sum(7.0) == 7.0
