"""The N>1 path of bench.py on CPU: world_size-2 gloo ranks (no GPU).

Each rank is an independent replica; the job's time is the slowest rank's and
its throughput counts the work of every rank."""
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


def _rank(rank, world, port, q):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms_local = 10.0 + 5.0 * rank            # rank 1 is the slow one
    ms, value = bench.aggregate_over_ranks(ms_local, 1e12, 4, world, dist, "cpu")
    q.put((rank, ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_max_time_and_sum_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in res:
        assert ms == 15.0
        # 2 replicas x 4 steps x 1e12 flops in 15 ms
        assert value == pytest.approx(2 * 4 * 1e12 / 15e-3 / 1e12)


def test_single_rank_is_plain_ratio():
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    ms, value = bench.aggregate_over_ranks(8.0, 1e13, 10, 1)
    assert ms == 8.0 and value == pytest.approx(1e13 * 10 / 8e-3 / 1e12)
