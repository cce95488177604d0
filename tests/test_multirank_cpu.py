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


def _counts_worker(rank, world, port, q):
    """Each rank holds a ragged shard of a seeded table (rank 2 none), counts its
    words' bits on the host and sums the counts through allreduce_counts."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import numpy as np

    import ibp_inputs as gen
    from lossless_bit_level_gb300.sharded import allreduce_counts
    words = gen.gnn_dense(1000).view(np.uint32)
    bounds = [0, 377, 1000, 1000]
    mine = words[bounds[rank]:bounds[rank + 1]]
    w32 = mine.ravel()
    counts = torch.tensor([int(((w32 >> np.uint32(j)) & np.uint32(1)).sum()) for j in range(32)],
                          dtype=torch.int64)
    total = allreduce_counts(counts, mine.size)
    q.put((rank, total, counts.tolist()))
    dist.barrier()
    dist.destroy_process_group()


def test_allreduce_counts_three_ranks():
    """The metadata exchange over gloo: summed counters equal the counts of the
    whole table and the element total is the table's, with one rank holding no rows."""
    import numpy as np

    import ibp_inputs as gen
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_counts_worker, args=(r, 3, port, q)) for r in range(3)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    words = gen.gnn_dense(1000).view(np.uint32).ravel()
    want = [int(((words >> np.uint32(j)) & np.uint32(1)).sum()) for j in range(32)]
    for rank, total, counts in res:
        assert total == words.size
        assert counts == want


def test_allreduce_counts_rejects_bad_buffer():
    from lossless_bit_level_gb300.sharded import allreduce_counts
    with pytest.raises(ValueError):
        allreduce_counts(torch.zeros(32, dtype=torch.int32), 1)


def _sharded_worker(rank, world, port, q):
    """sharded_meta's orchestration over gloo with the two device calls replaced by
    host stand-ins: the local count, the exchange, the finalize with the totals."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import numpy as np

    import ibp_inputs as gen
    import lossless_bit_level_gb300.sharded as sh
    seen = {}

    def fake_count(rows, counters, dtype=None, stream=None):
        w32 = rows.numpy().view(np.uint32).ravel()
        counters.copy_(torch.tensor([int(((w32 >> np.uint32(j)) & np.uint32(1)).sum())
                                     for j in range(32)], dtype=torch.int64))

    def fake_finalize(counters, n_elems, dtype, T, block_elems, meta, stream=None):
        seen.update(counters=counters.tolist(), n_elems=n_elems, T=T, B=block_elems)

    sh.meta_count, sh.meta_finalize = fake_count, fake_finalize
    words = gen.gnn_dense(600).view(np.int32)
    bounds = [0, 600, 600]  # rank 1 holds no rows
    mine = torch.from_numpy(np.ascontiguousarray(words[bounds[rank]:bounds[rank + 1]]))
    counters = torch.full((32,), -1, dtype=torch.int64)
    total = sh.sharded_meta(mine, 0.9, 32, torch.zeros(4, dtype=torch.int32), counters,
                            dtype=0)
    q.put((rank, total, seen))
    dist.barrier()
    dist.destroy_process_group()


def test_sharded_meta_two_ranks():
    import numpy as np

    import ibp_inputs as gen
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_sharded_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w32 = gen.gnn_dense(600).view(np.uint32).ravel()
    want = [int(((w32 >> np.uint32(j)) & np.uint32(1)).sum()) for j in range(32)]
    for rank, total, seen in res:
        assert total == w32.size == seen["n_elems"]
        assert seen["counters"] == want
        assert (seen["T"], seen["B"]) == (0.9, 32)
