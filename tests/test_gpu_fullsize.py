"""Parity at the full workload sizes, in the launch configuration bench.py times.

Per workload:
  * metadata: GPU vs oracle over the whole table or tensor;
  * compression: the slots, bitmask bits and per-row sizes of a random sample of rows
    against the oracle's own compression of the same rows with the same metadata;
  * decompress-gather: full index batches, every gathered row against the original
    row (exact; the codec is lossless) and against the oracle's gather of the sampled
    rows from the oracle's slots.
Tables are generated, checked and freed one at a time.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import ibp_inputs as gen
import lossless_bit_level_gb300 as ibp
import oracle
from codec_harness import GpuStore, gpu_compress, gpu_gather, gpu_meta, meta_tensor, meta_values, \
    to_torch

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def check_table(words: np.ndarray, dtype: int, T: float, B: int, batches, residencies,
                sample_rows: int = 4096, oracle_meta: bool = True, seed: int = 0,
                oracle_meta_future=None):
    """oracle_meta_future: the oracle's (mask, bitval) of ``words`` being computed in
    another thread (a concurrent.futures.Future), used instead of computing it here."""
    n, L = words.shape
    raw = L * words.dtype.itemsize
    rows_host = to_torch(words, "host")
    meta = gpu_meta(rows_host, dtype, T, B)
    mask, bitval, mdt, mb = meta_values(meta)
    assert (mdt, mb) == (dtype, B)
    if oracle_meta_future is not None:
        assert (mask, bitval) == oracle_meta_future.result()
    elif oracle_meta:
        assert (mask, bitval) == oracle.build_meta(words, T)
    # compress zero-copy from host rows into host slots (the bench's configuration)
    store = GpuStore(n, L, dtype, B, "host")
    gpu_compress(rows_host, meta, store)
    torch.cuda.synchronize()
    assert int(store.status.item()) == 0
    g = np.random.default_rng(seed)
    sample = np.unique(np.concatenate([g.integers(0, n, size=sample_rows), [0, n - 1]]))
    o_slots, o_bitmask, o_row_bits = oracle.compress(words[sample], B, mask, bitval)
    bm = store.bitmask.cpu().numpy().view(np.uint32)
    flags = (bm[sample // 32] >> (sample % 32).astype(np.uint32)) & 1
    o_flags = (o_bitmask[np.arange(sample.size) // 32] >>
               (np.arange(sample.size) % 32).astype(np.uint32)) & 1
    assert np.array_equal(flags, o_flags)
    rb = store.row_bits.cpu().numpy().view(np.uint32)[:n]
    assert np.array_equal(rb[sample], o_row_bits)
    gslots = store.slots[torch.from_numpy(sample)].numpy()
    used = np.where(o_flags == 1, 4 * ((o_row_bits.astype(np.int64) + 31) // 32), raw)
    for k in range(sample.size):
        assert np.array_equal(gslots[k, :used[k]], o_slots[k, :used[k]]), int(sample[k])
    # the last bitmask word has no bits past n_rows
    if n % 32:
        assert int(bm[-1]) >> (n % 32) == 0
    for where in residencies:
        if where == "device":
            dstore = GpuStore.__new__(GpuStore)
            dstore.__dict__.update(store.__dict__)
            dstore.slots = store.slots.to("cuda")
            use = dstore
        else:
            use = store
        for idx in batches:
            out, st = gpu_gather(use, meta, idx)
            assert st == 0
            got = out.cpu().numpy().view(words.dtype)
            assert np.array_equal(got, words[idx]), where
            # the oracle's gather of the sampled rows from the oracle's own slots
            pick = np.nonzero(np.isin(idx, sample))[0][:2048]
            if pick.size:
                pos = np.searchsorted(sample, idx[pick])
                o_out, rc = oracle.decompress_gather(o_slots, sample.size, L, words.dtype, B,
                                                     o_bitmask, mask, bitval, pos)
                assert rc == 0
                assert np.array_equal(got[pick], o_out)
            del out
        if where == "device":
            del dstore
        torch.cuda.empty_cache()
    return store


def test_gnn_dense_full():
    """2,000,000 x 128 FP32, T = 0.9, B = 32; 100,000 Zipf(1.0) indices, host and HBM."""
    words = gen.gnn_dense().view(np.uint32)
    batches = [gen.zipf_indices(words.shape[0], 100_000, 1.0, part=k, workload=gen.GNN_DENSE)
               for k in range(2)]
    check_table(words, ibp.FP32, 0.9, 32, batches, ("host", "device"))


def test_gnn_sparse_full():
    """500,000 x 512 FP32 binary, T = 0.9, B = 32; 100,000 uniform indices, host and HBM."""
    words = gen.gnn_sparse().view(np.uint32)
    batches = [gen.uniform_indices(words.shape[0], 100_000, part=k, workload=gen.GNN_SPARSE)
               for k in range(2)]
    check_table(words, ibp.FP32, 0.9, 32, batches, ("host", "device"))


def test_dlrm_all_tables_full():
    """26 tables x 1,000,000 x 128 FP32, per-table meta T = 0.95, B = 32; 65,536 Zipf(1.05)
    lookups per table, host and HBM. The oracle builds the metadata of every fourth
    table over the whole table (its slowest step); every table is checked otherwise."""
    for t in range(26):
        words = gen.dlrm_table(t).view(np.uint32)
        batches = [gen.zipf_indices(words.shape[0], 65_536, 1.05, part=t, workload=gen.DLRM)]
        check_table(words, ibp.FP32, 0.95, 32, batches, ("host", "device") if t < 2 else ("host",),
                    sample_rows=1024, oracle_meta=(t % 4 == 0), seed=t)
        del words
        torch.cuda.empty_cache()


_LLM_TENSORS = [*gen.LLM_MATRICES, "K", "V"]
_pool = None
_pending = {}  # layer -> {tensor name: Future of its words}


def _llm_pool() -> cf.ThreadPoolExecutor:
    global _pool
    if _pool is None:  # numpy's generators and the oracle's C calls release the GIL
        _pool = cf.ThreadPoolExecutor(max_workers=max(2, min(12, os.cpu_count() or 2)))
    return _pool


def _llm_layer_futures(layer: int) -> dict:
    if layer not in _pending:
        pool = _llm_pool()
        futs = {name: pool.submit(gen.llm_weight, layer, name) for name in gen.LLM_MATRICES}
        futs["K"] = pool.submit(gen.llm_kv, layer, 0)
        futs["V"] = pool.submit(gen.llm_kv, layer, 1)
        _pending[layer] = futs
    return _pending[layer]


@pytest.mark.parametrize("layer", range(gen.LLM_LAYERS))
def test_llm_layer_full(layer):
    """Every decoder layer at full size: the seven weight matrices and the K, V caches
    (8 x 4096 tokens x 4096 channels), per tensor T = 0.9, B = 64; the metadata of
    every tensor against the oracle's over the whole tensor, sampled slots against
    the oracle's, every row streamed in order from host slots (the K and V caches
    also from HBM) against the original. The next layer is generated in background
    threads while this one is checked."""
    futs = _llm_layer_futures(layer)
    if layer + 1 < gen.LLM_LAYERS:
        _llm_layer_futures(layer + 1)
    pool = _llm_pool()
    try:
        for name in _LLM_TENSORS:
            words = futs[name].result()
            o_meta = pool.submit(oracle.build_meta, words, 0.9)
            idx = np.arange(words.shape[0], dtype=np.int64)
            kv = name in ("K", "V")
            check_table(words, ibp.BF16, 0.9, 64, [idx], ("host", "device") if kv else ("host",),
                        sample_rows=1024 if kv else 512, seed=layer + (name == "V"),
                        oracle_meta_future=o_meta)
            del words
            futs[name] = None
            torch.cuda.empty_cache()
    finally:
        _pending.pop(layer, None)


def test_gnn_dense_variants_full():
    """The next-step variants on the full 2,000,000 x 128 dense GNN table:
    * saving-aware metadata: every candidate's score equals the stored bytes the GPU
      compression reports (ibp_query) for that candidate's mask, and the chosen one is
      the smallest; the candidate masks are the oracle's on a 200,000-row prefix's
      threshold family (same counts order) -- checked by recomputing the threshold
      mask from numpy bit counts of the whole table;
    * per-position metadata: the GPU arrays equal numpy bit counts column by column;
      rows compressed with them round-trip, sampled slots equal the oracle's;
    * sized and packed gathers of full batches equal the original rows."""
    words = gen.gnn_dense().view(np.uint32)
    n, L = words.shape
    T, B = 0.9, 32
    dev = torch.device("cuda")
    rows = to_torch(words, "host")
    # bit counts of the whole table (numpy, 64 positions at a time)
    ones = np.zeros(32, dtype=np.int64)
    col_ones = np.zeros((L, 32), dtype=np.int64)
    for r0 in range(0, n, 250_000):
        chunk = words[r0:r0 + 250_000]
        for j in range(32):
            b = (chunk >> np.uint32(j)) & np.uint32(1)
            col = b.sum(axis=0, dtype=np.int64)
            col_ones[:, j] += col
            ones[j] += col.sum()
    # saving-aware selection
    meta = torch.zeros(4, dtype=torch.int32, device=dev)
    scratch = torch.empty(ibp.meta_select_scratch_bytes() // 4, dtype=torch.int32, device=dev)
    cand = torch.zeros((ibp.MAX_MASK_CANDIDATES, 4), dtype=torch.int32, device=dev)
    ibp.build_meta_select(rows, T, B, meta, scratch, cand, dtype=ibp.FP32)
    torch.cuda.synchronize()
    cands = ibp.read_candidates(cand)
    N = n * L
    held = np.maximum(ones, N - ones)
    m0 = sum(1 << j for j in range(32) if float(held[j]) >= T * float(N))
    assert cands[0][0] == m0
    store = GpuStore(n, L, ibp.FP32, B, "host")
    for mk, bv, score in cands:
        m = meta_tensor(mk, bv, ibp.FP32, B)
        gpu_compress(rows, m, store)
        assert ibp.query(store.bitmask, store.row_bits, n, L, ibp.FP32).stored_bytes == score, \
            hex(mk)
    chosen = meta.cpu().numpy().view(np.uint32)
    assert int(chosen[0]) == min(cands, key=lambda c: (c[2], -bin(c[0]).count("1")))[0]
    # sized and packed gathers of the chosen store
    gpu_compress(rows, meta, store)
    idx = gen.zipf_indices(n, 100_000, 1.0, part=7, workload=gen.GNN_DENSE)
    it = torch.from_numpy(idx).to(dev)
    out = torch.zeros((idx.size, L), dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ibp.decompress_gather_sized(store.slots, n, L, ibp.FP32, B, store.bitmask, store.row_bits,
                                meta, it, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and np.array_equal(out.cpu().numpy().view(np.uint32), words[idx])
    offsets = torch.zeros(n + 1, dtype=torch.int64, device=dev)
    kscr = torch.empty(ibp.pack_scratch_bytes(n) // 8, dtype=torch.int64, device=dev)
    ibp.pack_offsets(store.bitmask, store.row_bits, n, L, ibp.FP32, offsets, kscr, status=st)
    total = int(offsets[-1].item())
    packed = torch.empty(total, dtype=torch.uint8, device=dev)
    kbm = torch.zeros_like(store.bitmask)
    ibp.pack(store.slots, n, L, ibp.FP32, store.bitmask, store.row_bits, offsets, packed, kbm,
             status=st)
    out.zero_()
    ibp.decompress_gather_packed(packed, offsets, n, L, ibp.FP32, B, kbm, meta, it, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and np.array_equal(out.cpu().numpy().view(np.uint32), words[idx])
    del packed
    # per-position metadata at T = 0.99
    Tp = 0.99
    pm = torch.zeros(L, dtype=torch.int32, device=dev)
    pb = torch.zeros(L, dtype=torch.int32, device=dev)
    pscr = torch.empty(ibp.meta_positions_scratch_bytes(L, ibp.FP32) // 8, dtype=torch.int64,
                       device=dev)
    ibp.build_meta_positions(rows, Tp, B, pm, pb, pscr, dtype=ibp.FP32)
    torch.cuda.synchronize()
    g_pm = pm.cpu().numpy().view(np.uint32)
    g_pb = pb.cpu().numpy().view(np.uint32)
    for e in range(L):
        c1 = col_ones[e]
        c0 = n - c1
        v = (c1 > c0).astype(np.int64)
        hv = np.where(v == 1, c1, c0)
        inv = hv.astype(np.float64) >= Tp * float(n)
        assert int(g_pm[e]) == sum(1 << j for j in range(32) if inv[j]), e
        assert int(g_pb[e]) == sum(1 << j for j in range(32) if inv[j] and v[j]), e
    ibp.compress_positions(rows, B, pm, pb, store.slots, store.bitmask, store.row_bits,
                           dtype=ibp.FP32)
    torch.cuda.synchronize()
    sample = np.unique(np.random.default_rng(3).integers(0, n, size=3000))
    o_slots, o_bm, o_rb = oracle.compress_positions(words[sample], B, g_pm, g_pb)
    rb = store.row_bits.cpu().numpy().view(np.uint32)
    assert np.array_equal(rb[sample], o_rb)
    gs = store.slots[torch.from_numpy(sample)].numpy()
    for k in range(sample.size):
        used = 4 * ((int(o_rb[k]) + 31) // 32) if (o_bm[k // 32] >> (k % 32)) & 1 else 4 * L
        assert np.array_equal(gs[k, :used], o_slots[k, :used]), int(sample[k])
    out.zero_()
    ibp.decompress_gather_positions(store.slots, n, L, ibp.FP32, B, store.bitmask, pm, pb, it, out,
                                    st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and np.array_equal(out.cpu().numpy().view(np.uint32), words[idx])
