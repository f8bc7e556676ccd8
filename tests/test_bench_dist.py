"""The N > 1 path of the benchmark on CPU: world-size-2 gloo ranks reduce their
step times to the slowest rank and report the whole job's tokens/s (weak
scaling: each rank runs its own layer on its own tokens, no data-path
collective)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.reduce_max(10.0 + 5.0 * rank)  # rank 1 is the slow one
    value = bench.job_throughput(8192, world, ms)
    out.put((rank, ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_reduction_takes_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in res:
        assert ms == 15.0
        assert value == pytest.approx(2 * 8192 / 0.015)


def test_single_process_reduction_is_identity():
    import bench
    assert bench.reduce_max(3.5) == 3.5
    assert bench.job_throughput(100, 1, 10.0) == pytest.approx(10000.0)
