"""GPU codec vs the oracle, element by element, on seeded inputs (needs a GPU)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ibp_inputs as gen
import lossless_bit_level_gb300 as ibp
import oracle
import pins
from codec_harness import (GpuStore, bitmask_np, compare_slots, from_torch, gpu_compress,
                           gpu_gather, gpu_meta, meta_tensor, meta_values, oracle_store,
                           row_bits_np, slots_np, to_torch, words_of)

pytestmark = pytest.mark.gpu

FP32, FP16, BF16, W8 = ibp.FP32, ibp.FP16, ibp.BF16, ibp.W8


def full_check(words: np.ndarray, dtype_code: int, T: float, B: int, idx: np.ndarray,
               where: str = "device", rows_where: str = "device"):
    """Meta, bitmask, row bits, slots and gathered rows against the oracle."""
    n, L = words.shape
    mask, bitval, o_slots, o_bitmask, o_row_bits = oracle_store(words, T, B)
    rows_t = to_torch(words, rows_where)
    meta = gpu_meta(rows_t, dtype_code, T, B)
    assert meta_values(meta) == (mask, bitval, dtype_code, B)
    store = GpuStore(n, L, dtype_code, B, where)
    gpu_compress(rows_t, meta, store)
    torch.cuda.synchronize()
    assert int(store.status.item()) == 0
    assert np.array_equal(bitmask_np(store), o_bitmask)
    assert np.array_equal(row_bits_np(store), o_row_bits)
    raw = L * words.dtype.itemsize
    compare_slots(slots_np(store), o_slots, o_bitmask, o_row_bits, raw)
    out, st = gpu_gather(store, meta, idx)
    assert st == 0
    o_out, rc = oracle.decompress_gather(o_slots, n, L, words.dtype, B, o_bitmask, mask, bitval, idx)
    assert rc == 0
    got = from_torch(out, words.dtype)
    assert np.array_equal(got, o_out)
    assert np.array_equal(got, words[idx])
    return store, meta, (mask, bitval, o_slots, o_bitmask, o_row_bits)


def test_tiny_fp32_full_config():
    """4096 x 128 FP32 N(0, 0.05), T = 0.9, B = 32, 1024 uniform indices, HBM."""
    words = words_of(gen.tiny_fp32())
    idx = gen.uniform_indices(words.shape[0], 1024, workload=gen.TINY)
    full_check(words, FP32, 0.9, 32, idx)


@pytest.mark.parametrize("where", ["device", "host"])
def test_gnn_dense_prefix(where):
    words = words_of(gen.gnn_dense(20_000))
    idx = gen.zipf_indices(words.shape[0], 5000, 1.0, workload=gen.GNN_DENSE)
    full_check(words, FP32, 0.9, 32, idx, where=where, rows_where=where)


@pytest.mark.parametrize("where", ["device", "host"])
def test_gnn_sparse_prefix(where):
    words = words_of(gen.gnn_sparse(4000))
    idx = gen.uniform_indices(words.shape[0], 3000, workload=gen.GNN_SPARSE)
    full_check(words, FP32, 0.9, 32, idx, where=where)


def test_dlrm_prefix():
    words = words_of(gen.dlrm_table(5, 20_000))
    idx = gen.zipf_indices(words.shape[0], 4096, 1.05, workload=gen.DLRM)
    full_check(words, FP32, 0.95, 32, idx, where="host")


@pytest.mark.parametrize("name", ["q", "down"])
def test_llm_weight_rows(name):
    words = gen.llm_weight(3, name, n_rows=300)
    idx = np.arange(words.shape[0], dtype=np.int64)
    full_check(words, BF16, 0.9, 64, idx, where="host")


def test_llm_kv_rows():
    words = gen.llm_kv(2, 1, n_rows=1000)
    idx = np.arange(words.shape[0], dtype=np.int64)[::-1].copy()
    full_check(words, BF16, 0.9, 64, idx)


@pytest.mark.parametrize("dtype_code,np_dt,B,L", [
    (FP32, np.uint32, 32, 96), (FP32, np.uint32, 64, 192), (FP32, np.uint32, 32, 1056),
    (FP16, np.uint16, 32, 32), (FP16, np.uint16, 32, 224), (BF16, np.uint16, 64, 64),
    (BF16, np.uint16, 32, 11008), (FP16, np.uint16, 64, 4160),
    # rows ending in a shorter block (row length not a multiple of B)
    (FP32, np.uint32, 32, 100), (FP32, np.uint32, 64, 1060), (FP16, np.uint16, 32, 72),
    (BF16, np.uint16, 64, 4104), (FP32, np.uint32, 64, 4), (BF16, np.uint16, 32, 8),
    # 8-bit element words (B = 32 is 8 lane words per block)
    (W8, np.uint8, 32, 128), (W8, np.uint8, 64, 256), (W8, np.uint8, 32, 48),
    (W8, np.uint8, 64, 4112), (W8, np.uint8, 32, 16), (W8, np.uint8, 64, 2048),
    # 32 KiB rows (the longest one CTA encodes) and just past it
    (FP32, np.uint32, 32, 8192), (FP32, np.uint32, 64, 8196), (BF16, np.uint16, 64, 16400)])
def test_shapes_and_ragged_tails(dtype_code, np_dt, B, L):
    """Several tiles, odd block counts (half-used last chunk for 16-bit B=32),
    multi-segment rows, rows not a multiple of 32 blocks, shorter last blocks
    (down to a one-vector row), 8-bit words."""
    g = np.random.default_rng(L * 7 + B)
    w = 8 * np.dtype(np_dt).itemsize
    n = 333
    base = g.integers(0, 1 << w, size=(n, L), dtype=np.uint64)
    hi = np.uint64(((1 << w) - 1) ^ ((1 << (w // 2 + 1)) - 1))
    flip = g.random(size=(n, L)) < 0.002
    words = np.where(flip, base, (base & ~hi) | (np.uint64(0x3F1E3F1E) & hi)).astype(np_dt)
    idx = np.concatenate([g.integers(0, n, size=500), [0, n - 1, 0, 0]]).astype(np.int64)
    full_check(words, dtype_code, 0.9, B, idx)


@pytest.mark.parametrize("dtype_code,np_dt,B,L,n", [
    (FP32, np.uint32, 32, 20480, 40),       # 80 KiB rows
    (BF16, np.uint16, 64, 65544, 12),       # 128 KiB rows, an 8-element last block
    (W8, np.uint8, 32, 1 << 20, 3),         # 1 MiB rows of 8-bit words
    (FP32, np.uint32, 64, 1 << 20, 2)])     # 4 MiB rows: the longest row accepted
def test_very_long_rows(dtype_code, np_dt, B, L, n):
    """Rows far past 64 KiB (participation bits of up to 32,768 blocks, most of them in
    vectors before the first payload word), host and HBM slots, compressed rows and
    raw ones (some rows are made incompressible), gathers of every row and repeats."""
    g = np.random.default_rng(L + B)
    w = 8 * np.dtype(np_dt).itemsize
    base = g.integers(0, 1 << w, size=(n, L), dtype=np.uint64)
    hi = np.uint64(((1 << w) - 1) ^ ((1 << (w // 2 + 1)) - 1))
    flip = g.random(size=(n, L)) < 0.0005
    words = np.where(flip, base, (base & ~hi) | (np.uint64(0x3F1E3F1E) & hi)).astype(np_dt)
    words[-1] = base[-1].astype(np_dt)  # one row of random words: stored raw
    idx = np.concatenate([np.arange(n), np.arange(n)[::-1], [0]]).astype(np.int64)
    for where in ("device", "host"):
        full_check(words, dtype_code, 0.9, B, idx, where=where)


@pytest.mark.parametrize("mask,bitval", [
    (0x00000000, 0x00000000),          # empty mask: every row raw
    (0xFFFFFFFF, 0x00000000),          # full mask: matching blocks are 0 bits
    (0x55555555, 0x41041041 & 0x55555555),  # 16 runs: generic deposit path
    (0x0F0F0F0F, 0x0A0B0C0D & 0x0F0F0F0F),  # 4 runs
    (0x7F800000, 0x3F800000),
])
@pytest.mark.parametrize("L", [128, 1600])
def test_forced_masks_fp32(mask, bitval, L):
    """Meta written directly (any mask is a valid code): compress + gather vs oracle,
    on short rows and on 6.4 KB rows (one CTA per row)."""
    g = np.random.default_rng(mask & 0xFFFF)
    n, B = 200, 32
    rnd = g.integers(0, 1 << 32, size=(n, L), dtype=np.uint64).astype(np.uint32)
    keep = g.random(size=(n, L)) < 0.995
    words = np.where(keep, (rnd & ~np.uint32(mask)) | np.uint32(bitval), rnd).astype(np.uint32)
    words[: n // 4] = rnd[: n // 4]  # some rows with no match at all
    o_slots, o_bitmask, o_row_bits = oracle.compress(words, B, mask, bitval)
    meta = meta_tensor(mask, bitval, FP32, B)
    store = GpuStore(n, L, FP32, B, "device")
    gpu_compress(to_torch(words, "device"), meta, store)
    torch.cuda.synchronize()
    assert np.array_equal(bitmask_np(store), o_bitmask)
    assert np.array_equal(row_bits_np(store), o_row_bits)
    compare_slots(slots_np(store), o_slots, o_bitmask, o_row_bits, L * 4)
    idx = g.integers(0, n, size=400)
    out, st = gpu_gather(store, meta, idx)
    assert st == 0
    assert np.array_equal(from_torch(out, np.uint32), words[idx])


@pytest.mark.parametrize("mask16", [0x7F80, 0xFFFF, 0x0000, 0x5555, 0x8001])
def test_forced_masks_bf16(mask16):
    g = np.random.default_rng(mask16)
    n, L, B = 150, 256, 64
    bitval = 0x3F80 & mask16
    rnd = g.integers(0, 1 << 16, size=(n, L), dtype=np.uint64).astype(np.uint16)
    keep = g.random(size=(n, L)) < 0.998
    words = np.where(keep, (rnd & ~np.uint16(mask16)) | np.uint16(bitval), rnd).astype(np.uint16)
    o_slots, o_bitmask, o_row_bits = oracle.compress(words, B, mask16, bitval)
    meta = meta_tensor(mask16, bitval, BF16, B)
    store = GpuStore(n, L, BF16, B, "host")
    gpu_compress(to_torch(words, "host"), meta, store)
    torch.cuda.synchronize()
    assert np.array_equal(bitmask_np(store), o_bitmask)
    assert np.array_equal(row_bits_np(store), o_row_bits)
    compare_slots(slots_np(store), o_slots, o_bitmask, o_row_bits, L * 2)
    idx = g.integers(0, n, size=300)
    out, st = gpu_gather(store, meta, idx)
    assert st == 0
    assert np.array_equal(from_torch(out, np.uint16), words[idx])


# masks whose matching lane words keep 8, 16 or 24 bits, in at most four runs with bit
# 0 kept: long rows take the compressor's 16-byte path for them
WHOLE_WORD_FIELDS = [
    (FP32, np.uint32, 0xFFFFFF00, 1000), (FP32, np.uint32, 0xFFFF0000, 1000),
    (FP32, np.uint32, 0x7F800000, 1000),
    (BF16, np.uint16, 0x7FF8, 2056), (BF16, np.uint16, 0x7F80, 2056),
    (BF16, np.uint16, 0x7800, 2056),
    (W8, np.uint8, 0xFC, 4112), (W8, np.uint8, 0xF0, 4112), (W8, np.uint8, 0xC0, 4112),
]


@pytest.mark.parametrize("B", [32, 64])
@pytest.mark.parametrize("dtype_code,np_dt,mask,L", WHOLE_WORD_FIELDS)
def test_whole_word_fields_long_rows(dtype_code, np_dt, mask, L, B):
    """Rows over 2 KiB (a ragged last block, a partial last step) with fields of 8, 16
    or 24 bits per lane word: blocks matching and not within a step, rows that never
    match, rows that match but save nothing; slots, bitmask and row sizes vs the
    oracle, then the gather."""
    g = np.random.default_rng(mask * 7 + B)
    n = 96
    bits = np.dtype(np_dt).itemsize * 8
    bitval = (0x5A5A5A5A & mask) & ((1 << bits) - 1)
    rnd = g.integers(0, 1 << bits, size=(n, L), dtype=np.uint64).astype(np_dt)
    keep = g.random(size=(n, L)) < 0.997
    words = np.where(keep, (rnd & ~np_dt(mask)) | np_dt(bitval), rnd).astype(np_dt)
    words[: n // 8] = rnd[: n // 8]  # no match at all
    lw = L // 8
    words[n // 8: n // 4, :lw] = rnd[n // 8: n // 4, :lw]  # a raw first stretch
    o_slots, o_bitmask, o_row_bits = oracle.compress(words, B, mask, bitval)
    meta = meta_tensor(mask, bitval, dtype_code, B)
    store = GpuStore(n, L, dtype_code, B, "device")
    gpu_compress(to_torch(words, "device"), meta, store)
    torch.cuda.synchronize()
    assert int(store.status.item()) == 0
    assert np.array_equal(bitmask_np(store), o_bitmask)
    assert np.array_equal(row_bits_np(store), o_row_bits)
    compare_slots(slots_np(store), o_slots, o_bitmask, o_row_bits, L * np.dtype(np_dt).itemsize)
    idx = g.integers(0, n, size=300)
    out, st = gpu_gather(store, meta, idx)
    assert st == 0
    assert np.array_equal(from_torch(out, np_dt), words[idx])


@pytest.mark.parametrize("w", [32, 16, 8])
def test_special_values_round_trip(w):
    g = np.random.default_rng(w)
    sp = np.array(pins.special_words(w), dtype={32: np.uint32, 16: np.uint16, 8: np.uint8}[w])
    n, L = 256, 128
    words = sp[g.integers(0, sp.size, size=(n, L))]
    words[: n // 2] = np.where(g.random(size=(n // 2, L)) < 0.97, sp[3], words[: n // 2])
    dtype_code = {32: FP32, 16: FP16, 8: W8}[w]
    for T in (0.0, 0.6, 0.95, 1.0):
        idx = g.integers(0, n, size=512)
        full_check(words, dtype_code, T, 32, idx)


def test_gpu_decodes_oracle_slots():
    """The decoder alone: slots written by the oracle, gathered by the GPU."""
    words = words_of(gen.gnn_sparse(2000))
    mask, bitval, o_slots, o_bitmask, o_row_bits = oracle_store(words, 0.9, 32)
    n, L = words.shape
    store = GpuStore(n, L, FP32, 32, "host")
    store.slots.copy_(torch.from_numpy(o_slots))
    store.bitmask.copy_(torch.from_numpy(o_bitmask.view(np.int32)))
    meta = meta_tensor(mask, bitval, FP32, 32)
    idx = gen.uniform_indices(n, 2500, workload=gen.GNN_SPARSE)
    out, st = gpu_gather(store, meta, idx)
    assert st == 0
    assert np.array_equal(from_torch(out, np.uint32), words[idx])


def test_error_status_and_edge_cases():
    words = words_of(gen.tiny_fp32(256))
    n, L = words.shape
    mask, bitval, o_slots, o_bitmask, o_row_bits = oracle_store(words, 0.9, 32)
    rows_t = to_torch(words, "device")
    meta = gpu_meta(rows_t, FP32, 0.9, 32)
    store = GpuStore(n, L, FP32, 32, "device")
    gpu_compress(rows_t, meta, store)
    # out-of-range index: row skipped, status INDEX, other rows still decoded
    sentinel = torch.full((3, L), -7, dtype=torch.int32, device="cuda")
    out, st = gpu_gather(store, meta, np.array([5, n, -1], dtype=np.int64), out=sentinel)
    assert st == ibp.ERR_INDEX
    got = from_torch(out, np.uint32)
    assert np.array_equal(got[0], words[5])
    assert np.all(got[1:] == np.uint32(0xFFFFFFF9))
    # corrupt header: clear the participation bits of a compressed row
    bm = bitmask_np(store)
    r = next(r for r in range(n) if (bm[r // 32] >> (r % 32)) & 1)
    store.slots[r, 0] = store.slots[r, 0] & 0xF0
    sentinel = torch.full((1, L), -7, dtype=torch.int32, device="cuda")
    out, st = gpu_gather(store, meta, np.array([r], dtype=np.int64), out=sentinel)
    assert st == ibp.ERR_CORRUPT
    assert np.all(from_torch(out, np.uint32) == np.uint32(0xFFFFFFF9))
    # empty gather: no-op, no launch
    out, st = gpu_gather(store, meta, np.zeros(0, dtype=np.int64))
    assert st == 0 and out.shape == (0, L)
    # metadata that disagrees with the call: status META, nothing written
    wrong = meta_tensor(mask, bitval, BF16, 32)
    sentinel = torch.full((1, L), -7, dtype=torch.int32, device="cuda")
    out, st = gpu_gather(store, wrong, np.array([0], dtype=np.int64), out=sentinel)
    assert st == ibp.ERR_META
    # argument errors are returned before any launch
    with pytest.raises(ibp.IBPError) as e:
        ibp.decompress_gather(store.slots, n, L, FP32, 48, store.bitmask, meta,
                              torch.zeros(1, dtype=torch.int64, device="cuda"),
                              torch.zeros((1, L), dtype=torch.int32, device="cuda"))
    assert e.value.code in (ibp.ERR_ARG, ibp.ERR_UNSUPPORTED)
    pageable = torch.zeros((n, store.slot_bytes), dtype=torch.uint8)
    with pytest.raises(ibp.IBPError) as e:
        ibp.decompress_gather(pageable, n, L, FP32, 32, store.bitmask, meta,
                              torch.zeros(1, dtype=torch.int64, device="cuda"),
                              torch.zeros((1, L), dtype=torch.int32, device="cuda"))
    assert e.value.code == ibp.ERR_ARG


def test_query_stats():
    """ibp_query (host output, synchronising) and ibp_query_async (device output)
    against the oracle's totals, on the current stream and on a side stream."""
    words = words_of(gen.gnn_dense(5000))
    n, L = words.shape
    mask, bitval, o_slots, o_bitmask, o_row_bits = oracle_store(words, 0.9, 32)
    rows_t = to_torch(words, "device")
    meta = gpu_meta(rows_t, FP32, 0.9, 32)
    store = GpuStore(n, L, FP32, 32, "device")
    gpu_compress(rows_t, meta, store)
    stored = oracle.stored_bytes(o_row_bits, o_bitmask, L * 4)
    flags = (o_bitmask[np.arange(n) // 32] >> (np.arange(n) % 32).astype(np.uint32)) & 1
    expect = (n, int(flags.sum()), n * L * 4, int(stored.sum()),
              int(o_row_bits.astype(np.int64).sum()))

    def fields(st):
        return (st.n_rows, st.n_compressed, st.raw_bytes, st.stored_bytes, st.total_bits)

    torch.cuda.synchronize()
    assert fields(ibp.query(store.bitmask, store.row_bits, n, L, FP32)) == expect
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    assert fields(ibp.query(store.bitmask, store.row_bits, n, L, FP32, stream=side)) == expect
    stats_t = torch.full((10,), -1, dtype=torch.int32, device="cuda")
    ibp.query_async(store.bitmask, store.row_bits, n, L, FP32, stats_t)
    assert fields(ibp.read_stats(stats_t)) == expect
    # a prefix of the store, and an empty one (null arrays allowed)
    k = 1234
    o_k = oracle.stored_bytes(o_row_bits[:k], o_bitmask, L * 4)
    st = ibp.query(store.bitmask, store.row_bits, k, L, FP32)
    assert (st.n_rows, st.n_compressed, st.stored_bytes) == (k, int(flags[:k].sum()),
                                                              int(o_k.sum()))
    assert fields(ibp.query(None, None, 0, L, FP32)) == (0, 0, 0, 0, 0)
    with pytest.raises(ibp.IBPError) as e:
        ibp.query(store.bitmask, store.row_bits, n, L, 7)
    assert e.value.code == ibp.ERR_DTYPE


def test_meta_from_host_rows_matches():
    words = gen.llm_kv(4, 0, n_rows=2048)
    mask, bitval = oracle.build_meta(words, 0.9)
    meta = gpu_meta(to_torch(words, "host"), BF16, 0.9, 64)
    assert meta_values(meta) == (mask, bitval, BF16, 64)


def test_probe_read_checksum():
    g = np.random.default_rng(3)
    a = g.integers(0, 1 << 32, size=1 << 16, dtype=np.uint64).astype(np.uint32)
    exp = int(np.bitwise_xor.reduce(a))
    sink = torch.zeros((2,), dtype=torch.int32, device="cuda")
    for where in ("device", "host"):
        ibp.probe_read(to_torch(a, where), sink)
        torch.cuda.synchronize()
        got = int(sink.cpu().numpy().view(np.uint64)[0])
        assert got == exp


@pytest.mark.parametrize("where", ["device", "host"])
def test_gather_in_cuda_graph(where):
    """A gather captured once in a CUDA graph and replayed on new index contents."""
    words = words_of(gen.gnn_dense(8000))
    n, L = words.shape
    rows_t = to_torch(words, "device")
    meta = gpu_meta(rows_t, FP32, 0.9, 32)
    store = GpuStore(n, L, FP32, 32, where)
    gpu_compress(rows_t, meta, store)
    idx = torch.zeros(3000, dtype=torch.int64, device="cuda")
    out = torch.zeros((3000, L), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ibp.decompress_gather(store.slots, n, L, FP32, 32, store.bitmask, meta, idx, out, status)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ibp.decompress_gather(store.slots, n, L, FP32, 32, store.bitmask, meta, idx, out, status,
                              stream=s)
    for k in range(3):
        ix = gen.zipf_indices(n, 3000, 1.0, part=50 + k, workload=gen.GNN_DENSE)
        idx.copy_(torch.from_numpy(ix))
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert np.array_equal(out.cpu().numpy().view(np.uint32), words[ix])


def test_concurrent_host_threads():
    """Four host threads, each with its own stream, gather from one store at once
    (the library keeps only per-device lookups that are filled once, under a lock)."""
    import threading
    words = words_of(gen.gnn_dense(6000))
    n, L = words.shape
    rows_t = to_torch(words, "device")
    meta = gpu_meta(rows_t, FP32, 0.9, 32)
    store = GpuStore(n, L, FP32, 32, "host")
    gpu_compress(rows_t, meta, store)
    torch.cuda.synchronize()
    errors = []

    def work(k):
        try:
            s = torch.cuda.Stream()
            g = np.random.default_rng(100 + k)
            for _ in range(20):
                ix = g.integers(0, n, size=777)
                idx = torch.from_numpy(ix).cuda()
                out = torch.zeros((ix.size, L), dtype=torch.int32, device="cuda")
                st = torch.zeros(1, dtype=torch.int32, device="cuda")
                torch.cuda.current_stream().synchronize()
                ibp.decompress_gather(store.slots, n, L, FP32, 32, store.bitmask, meta, idx, out,
                                      st, stream=s)
                s.synchronize()
                assert int(st.item()) == 0
                assert np.array_equal(out.cpu().numpy().view(np.uint32), words[ix])
        except Exception as e:  # collected and re-raised in the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(k,)) for k in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[0]


@pytest.mark.parametrize("where", ["host", "device"])
@pytest.mark.parametrize("name", ["dense", "sparse", "kv", "w8_tail"])
def test_sized_gather(where, name):
    """The sized gather (row sizes from row_bits, only the used prefix staged)
    against the oracle and the original rows; a row size that disagrees with the
    row's header is reported as corrupt and the row left untouched."""
    if name == "dense":
        words, code, T, B = words_of(gen.gnn_dense(8000)), FP32, 0.9, 32
    elif name == "sparse":
        words, code, T, B = words_of(gen.gnn_sparse(3000)), FP32, 0.9, 32
    elif name == "kv":
        words, code, T, B = gen.llm_kv(2, 1, n_rows=600), BF16, 0.9, 64
    else:
        g = np.random.default_rng(8)
        base = g.integers(0, 256, size=(700, 4112), dtype=np.uint64)
        words = np.where(g.random(size=base.shape) < 0.003, base,
                         (base & np.uint64(0x1F)) | np.uint64(0x40)).astype(np.uint8)
        code, T, B = W8, 0.9, 64
    n, L = words.shape
    mask, bitval, o_slots, o_bitmask, o_row_bits = oracle_store(words, T, B)
    rows_t = to_torch(words, where)
    meta = gpu_meta(rows_t, code, T, B)
    store = GpuStore(n, L, code, B, where)
    gpu_compress(rows_t, meta, store)
    g = np.random.default_rng(n)
    ix = np.concatenate([g.integers(0, n, size=2000), [0, n - 1]]).astype(np.int64)
    wdt = {4: torch.int32, 2: torch.int16, 1: torch.uint8}[words.dtype.itemsize]
    out = torch.zeros((ix.size, L), dtype=wdt, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ibp.decompress_gather_sized(store.slots, n, L, code, B, store.bitmask, store.row_bits, meta,
                                torch.from_numpy(ix).cuda(), out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = from_torch(out, words.dtype)
    o_out, rc = oracle.decompress_gather(o_slots, n, L, words.dtype, B, o_bitmask, mask, bitval, ix)
    assert rc == 0 and np.array_equal(got, o_out) and np.array_equal(got, words[ix])
    # a compressed row whose recorded size is cut below its stream is corrupt
    comp_rows = [r for r in range(n) if (o_bitmask[r // 32] >> (r % 32)) & 1
                 and o_row_bits[r] > 160]
    if comp_rows:
        r = comp_rows[0]
        other = (r + 1) % n
        bad_bits = store.row_bits.clone()
        bad_bits[r] = 64  # 8 bytes: rounds to one 16-byte piece
        sentinel = torch.full((2, L), 5, dtype=wdt, device="cuda")
        st.zero_()
        ibp.decompress_gather_sized(store.slots, n, L, code, B, store.bitmask, bad_bits, meta,
                                    torch.tensor([r, other], dtype=torch.int64, device="cuda"),
                                    sentinel, st)
        torch.cuda.synchronize()
        assert int(st.item()) == ibp.ERR_CORRUPT
        res = from_torch(sentinel, words.dtype)
        assert np.all(res[0] == 5) and np.array_equal(res[1], words[other])


@pytest.mark.parametrize("n_tables", [5, 70])
def test_batched_gather_tables(n_tables):
    """One call gathering from many tables (each its own store, metadata, indices and
    output; some host-resident, one job with no indices, one with a bad index), more
    than 64 jobs split into launches; every job against the oracle."""
    g = np.random.default_rng(n_tables)
    L, B, T = 128, 32, 0.95
    jobs, expect, bad_job = [], [], None
    for t in range(n_tables):
        words = words_of(gen.dlrm_table(t % 26, 2000 + 37 * t))
        n = words.shape[0]
        where = "host" if t % 3 == 0 else "device"
        rows_t = to_torch(words, where)
        meta = gpu_meta(rows_t, FP32, T, B)
        store = GpuStore(n, L, FP32, B, where)
        gpu_compress(rows_t, meta, store)
        k = 0 if t == 1 else int(g.integers(1, 900))
        ix = g.integers(0, n, size=k).astype(np.int64)
        if t == 2:
            ix[0] = n + 5  # out of range: skipped, reported
            bad_job = t
        out = torch.full((max(k, 1), L), 9, dtype=torch.int32, device="cuda")
        jobs.append((store.slots, n, store.bitmask, meta, torch.from_numpy(ix).cuda(), out, store))
        expect.append((words, ix))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ibp.decompress_gather_batched([j[:6] for j in jobs], L, FP32, B, status)
    torch.cuda.synchronize()
    assert int(status.item()) == ibp.ERR_INDEX
    for t, ((words, ix), job) in enumerate(zip(expect, jobs)):
        got = job[5].cpu().numpy().view(np.uint32)[: ix.size]
        if t == bad_job:
            assert np.all(got[0] == 9)
            assert np.array_equal(got[1:], words[ix[1:]])
        else:
            assert np.array_equal(got, words[ix]), t
