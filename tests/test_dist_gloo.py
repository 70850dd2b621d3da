"""Multi-rank host path of the benchmark (replicas) on CPU with gloo, world
size 2: max-over-ranks timing and whole-job throughput."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = 10.0 + 5.0 * rank          # rank 1 is the slow one
        ms, gbps = bench.aggregate(ms_local, 1_000_000_000, world)
        bench.barrier()
        q.put((rank, ms, gbps))
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, gbps in res:
        assert ms == pytest.approx(15.0)
        assert gbps == pytest.approx(2e9 / 15e-3 / 1e9)


def test_single_process_is_identity():
    import bench
    ms, gbps = bench.aggregate(4.0, 8_000_000, 1)
    assert ms == 4.0 and gbps == pytest.approx(2.0)
