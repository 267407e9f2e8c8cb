"""The N>1 bench path on CPU: two gloo ranks agree on the slowest rank's
timed interval and on the whole-job (weak-scaling) throughput."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_us = 30.0 + 5.0 * rank          # rank 1 is the slow one
    slowest = bench.reduce_max_over_ranks(local_us)
    value = bench.whole_job_gbs(134_234_112, world, slowest)
    dist.barrier()
    results[rank] = (slowest, value)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_interval():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert results[0] == results[1]
    slowest, value = results[0]
    assert slowest == 35.0
    assert abs(value - 2 * 134_234_112 / 35e-6 / 1e9) < 1e-6


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max_over_ranks(12.5) == 12.5
    assert abs(bench.whole_job_gbs(1_000_000, 1, 1.0) - 1000.0) < 1e-9
