"""The bench's multi-rank accounting on CPU: world size 2 over gloo (no GPU).

Ranks are independent replicas (no collective on the data path); the job's step
time is the slowest rank's and its throughput the sum of every rank's bytes over
that time."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t_local = [0.002, 0.003][rank]
    bytes_local = [1e9, 2e9][rank]
    t, gbs = bench.job_throughput(t_local, bytes_local, dist, torch.device("cpu"))
    dist.barrier()
    q.put((rank, t, gbs))
    dist.destroy_process_group()


def test_job_throughput_two_ranks():
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
    for rank, t, gbs in res:
        assert t == pytest.approx(0.003)
        assert gbs == pytest.approx(3e9 / 0.003 / 1e9)


def test_job_throughput_single_process():
    import bench
    t, gbs = bench.job_throughput(0.004, 2e9)
    assert t == 0.004 and gbs == pytest.approx(500.0)
