"""The multi-rank (replica) path of bench.py on CPU with the gloo backend:
each rank times its own replica; the job time is the slowest rank's and the
job throughput counts every rank's arena."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, local = bench.dist_info()
    assert (ws, r, local) == (world, rank, rank)
    ms = bench.max_over_ranks(10.0 + 3.0 * rank, torch.device("cpu"))
    dist.barrier()
    q.put((rank, ms, bench.job_gradient_gbs(1000, ws, ms)))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_job_throughput(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    slowest = 10.0 + 3.0 * (world - 1)
    for rank, ms, gbs in res:
        assert ms == slowest
        assert gbs == pytest.approx(world * 4.0 * 1000 / (slowest * 1e-3) / 1e9)


def test_single_process_is_its_own_max():
    import bench
    assert bench.max_over_ranks(7.5, torch.device("cpu")) == 7.5
