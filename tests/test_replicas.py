"""Replica aggregation of bench.py over two gloo ranks on CPU (the N > 1 path without GPUs)."""
import os
import socket

import pytest

pytestmark = pytest.mark.cpu


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    times = {0: 0.010, 1: 0.013}
    q.put((rank, bench.aggregate_replicas(times[rank], 1.5e9, dist)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregate_takes_slowest_rank_and_sums_bytes():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        gbps, t = res[r]
        assert t == pytest.approx(0.013)
        assert gbps == pytest.approx(2 * 1.5e9 / 0.013 / 1e9)


def test_single_process_aggregate():
    import bench
    gbps, t = bench.aggregate_replicas(0.002, 1e9, None)
    assert t == 0.002 and gbps == pytest.approx(500.0)
