"""The N>1 host logic of bench.py on CPU: two gloo ranks, independent replicas,
the job's time is the slowest rank's and its value counts every rank's work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = 10.0 + 5.0 * rank  # rank 1 is slower
    ms_max, tflops = bench.aggregate(ms, 2e12, world, torch.device("cpu"))
    q.put((rank, ms_max, tflops))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas_take_max_time():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, tflops in out:
        assert ms_max == 15.0
        assert tflops == pytest.approx(2e12 * 2 / 15e-3 / 1e12)


def test_single_rank_is_identity():
    import bench

    ms_max, tf = bench.aggregate(4.0, 8e12, 1, torch.device("cpu"))
    assert ms_max == 4.0 and tf == pytest.approx(2000.0)
