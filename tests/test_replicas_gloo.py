"""Multi-rank host logic of bench.py on CPU: two gloo ranks, each a replica with its
own time; the job time is the slowest rank's and the value counts every rank's rows."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    my_ms = [120.0, 150.0][rank]
    ms = bench.max_over_ranks(my_ms, world, "cpu")
    value = bench.job_rows_per_s(15435 * 50 * 5, world, ms)
    q.put((rank, ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in res:
        assert ms == 150.0
        assert abs(value - 2 * 15435 * 50 * 5 / 0.150) < 1e-6 * value


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(7.5, 1, "cpu") == 7.5
    assert bench.job_rows_per_s(1000, 1, 500.0) == 2000.0
