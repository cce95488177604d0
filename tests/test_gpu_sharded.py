"""Metadata of rows split over several holders, on the GPU against the oracle.

Bit counts of disjoint row sets add up ("Reducing the GPU Memory Bottleneck with
Lossless Compression for ML -- Extended", technical summary, "Core algorithm",
preprocessing), so counting each shard with ``ibp_meta_count``, summing the
counters and applying ``ibp_meta_finalize`` to the sums must give the oracle's
metadata of the union of the shards. Shards are cut at ragged row boundaries and
held in HBM or in page-locked host memory; one case goes through the
``torch.distributed`` exchange with a one-rank NCCL group."""
from __future__ import annotations

import socket

import numpy as np
import pytest
import torch

import ibp_inputs as gen
import lossless_bit_level_gb300 as ibp
import oracle
from codec_harness import GpuStore, gpu_meta, meta_values, to_torch

pytestmark = pytest.mark.gpu

FP32, FP16, BF16, W8 = ibp.FP32, ibp.FP16, ibp.BF16, ibp.W8


def split_meta(words: np.ndarray, cuts: list[int], code: int, T: float, B: int,
               where: str = "device"):
    bounds = [0] + cuts + [words.shape[0]]
    total = torch.zeros(32, dtype=torch.int64, device="cuda")
    n_elems = 0
    for a, b in zip(bounds[:-1], bounds[1:]):
        c = torch.full((32,), -1, dtype=torch.int64, device="cuda")  # overwritten
        if b > a:
            ibp.meta_count(to_torch(words[a:b], where), c, dtype=code)
        else:
            c.zero_()
        total += c
        n_elems += (b - a) * words.shape[1]
    meta = torch.zeros(4, dtype=torch.int32, device="cuda")
    ibp.meta_finalize(total, n_elems, code, T, B, meta)
    torch.cuda.synchronize()
    return meta_values(meta), total.cpu().numpy()


def bit_counts(words: np.ndarray) -> np.ndarray:
    """Per-position 1-counts of the rows' 32-bit words (brute force on the host)."""
    w32 = np.ascontiguousarray(words).view(np.uint32).ravel()
    return np.array([int(((w32 >> np.uint32(j)) & np.uint32(1)).sum()) for j in range(32)])


@pytest.mark.parametrize("where", ["device", "host"])
@pytest.mark.parametrize("T", [0.5, 0.9, 0.99, 1.0])
def test_gnn_dense_shards(where, T):
    words = gen.gnn_dense(20_000).view(np.uint32)
    (mask, bitval, dt, B), counts = split_meta(words, [7001, 12_999, 13_000], FP32, T, 32,
                                               where)
    assert np.array_equal(counts, bit_counts(words))
    assert (mask, bitval) == oracle.build_meta(words, T)
    assert (dt, B) == (FP32, 32)
    # one holder: the pair equals the one-call build
    whole = gpu_meta(to_torch(words, where), FP32, T, 32)
    assert meta_values(whole) == (mask, bitval, FP32, 32)


@pytest.mark.parametrize("code,B", [(BF16, 64), (FP16, 32), (W8, 64)])
def test_narrow_words_shards(code, B):
    if code == W8:
        x = gen.gnn_sparse(3000, 512)
        words = (x.view(np.uint32) >> np.uint32(23)).astype(np.uint8)
    else:
        words = gen.llm_weight(0, "q", n_rows=3000)
        if code == FP16:
            words = words ^ np.uint16(0x0100)
    for T in (0.6, 0.95):
        (mask, bitval, dt, b), counts = split_meta(words, [1, 1499, 2999], code, T, B)
        assert np.array_equal(counts, bit_counts(words))
        assert (mask, bitval) == oracle.build_meta(words, T)
        assert (dt, b) == (code, B)


def test_empty_shard_and_tie():
    """A holder with no rows adds nothing; an exact 50/50 split of a position keeps 0
    and is invariant only at T <= 0.5."""
    rows = np.zeros((64, 128), dtype=np.uint32)
    rows[:32, :] |= np.uint32(1 << 5)  # bit 5: half the elements 1
    for T in (0.5, 0.5000001):
        (mask, bitval, _, _), _ = split_meta(rows, [0, 0, 32], FP32, T, 32)
        assert (mask, bitval) == oracle.build_meta(rows, T)
        assert bool(mask >> 5 & 1) == (T <= 0.5) and not (bitval >> 5 & 1)


def test_finalize_rejects_counts_above_element_count():
    """Counters summed over two holders finalized with one holder's element count:
    no such set of elements exists, so the metadata comes back invalid (no invariant
    position, dtype IBP_META_INVALID), ERR_META is recorded, and compression given
    that metadata reports ERR_META instead of storing every row raw."""
    words = gen.gnn_dense(4000).view(np.uint32)
    (_, _, _, _), total = split_meta(words, [2000], FP32, 0.9, 32)
    counters = torch.from_numpy(total.astype(np.int64)).cuda()
    meta = torch.zeros(4, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # the first holder's element count with the summed counters: some position has
    # more ones than elements
    n_one = 2000 * words.shape[1]
    assert int(total.max()) > n_one
    ibp.meta_finalize(counters, n_one, FP32, 0.9, 32, meta, status)
    torch.cuda.synchronize()
    assert int(status.item()) == ibp.ERR_META
    m = meta.cpu().numpy().view(np.uint32)
    assert (int(m[0]), int(m[1]), int(m[2]), int(m[3])) == (0, 0, 0xFFFFFFFF, 32)
    # the right count on the same counters gives the oracle's metadata, status untouched
    status.zero_()
    ibp.meta_finalize(counters, words.size, FP32, 0.9, 32, meta, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert meta_values(meta) == (*oracle.build_meta(words, 0.9), FP32, 32)
    # a compression given the refused metadata reports it
    bad = torch.tensor([0, 0, -1, 32], dtype=torch.int32, device="cuda")
    n, L = words.shape
    store = GpuStore(n, L, FP32, 32, "device")
    ibp.compress(to_torch(words, "device"), 32, bad, store.slots, store.bitmask, store.row_bits,
                 store.status, dtype=FP32)
    torch.cuda.synchronize()
    assert int(store.status.item()) == ibp.ERR_META


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_sharded_meta_through_nccl():
    import torch.distributed as dist
    from lossless_bit_level_gb300.sharded import sharded_meta
    assert not dist.is_initialized()
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0,
                            world_size=1, device_id=torch.device("cuda", 0))
    try:
        words = gen.gnn_dense(5000).view(np.uint32)
        meta = torch.zeros(4, dtype=torch.int32, device="cuda")
        counters = torch.zeros(32, dtype=torch.int64, device="cuda")
        total = sharded_meta(to_torch(words, "device"), 0.9, 64, meta, counters, dtype=FP32)
        torch.cuda.synchronize()
        assert total == words.size
        assert np.array_equal(counters.cpu().numpy(), bit_counts(words))
        assert meta_values(meta) == (*oracle.build_meta(words, 0.9), FP32, 64)
        # a holder with no rows, called on a stream that is not the current one: the
        # counters are cleared on that stream, before the exchange reads them
        counters.fill_(-7)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        empty = torch.empty((0, words.shape[1]), dtype=torch.int32, device="cuda")
        with pytest.raises(ValueError):
            sharded_meta(empty, 0.9, 64, meta, counters, dtype=FP32, stream=side)
        torch.cuda.synchronize()
        assert np.array_equal(counters.cpu().numpy(), np.zeros(32, dtype=np.int64))
    finally:
        dist.destroy_process_group()
