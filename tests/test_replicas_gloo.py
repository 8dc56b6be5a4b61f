"""Multi-process host logic of bench.py on the CPU (gloo, world size 2):
every rank runs its own replica, the job's time is the slowest rank's and its
work is the sum over ranks.  No GPU is involved."""
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


def _worker(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench

    ranks = bench.Ranks(world)
    my_time = 1.0 + rank  # rank 1 is the slow one
    slowest = ranks.max(my_time)
    total_steps = ranks.sum(10.0)
    ranks.barrier()
    value = bench.replica_throughput(2e12, 10, [slowest] * world)
    out.put((rank, slowest, total_steps, value))
    ranks.close()


def test_two_ranks_take_the_slowest_time_and_sum_the_work():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, total, value in results:
        assert slowest == 2.0
        assert total == 20.0
        # 2 ranks x 10 steps x 2e12 flop over 2 s = 20 TFLOP/s
        assert value == pytest.approx(20.0)


def test_single_process_reduction_is_identity():
    import bench

    assert bench.reduce_over_ranks(None, 3.5, "max") == 3.5
    assert bench.replica_throughput(1e12, 4, [2.0]) == pytest.approx(2.0)
