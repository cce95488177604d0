"""De-duplicated decompress-gather on the GPU against the oracle (needs a GPU).

Every case builds the store with the GPU codec, gathers with
ibp_decompress_gather_dedup and compares every output row with the original row,
with the oracle's gather from the oracle's own slots, and with the plain GPU
gather. Index lists: Zipf-skewed (most positions repeat a few hot rows), all
distinct, one row repeated, bad indices mixed in; slots in HBM and in host memory;
32-, 16- and 8-bit words; rows served by the team kernel and by the
warp-specialised kernel."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ibp_inputs as gen
import lossless_bit_level_gb300 as ibp
import oracle
from codec_harness import GpuStore, from_torch, gpu_compress, gpu_gather, gpu_meta, oracle_store, \
    to_torch, words_of

pytestmark = pytest.mark.gpu

FP32, FP16, BF16, W8 = ibp.FP32, ibp.FP16, ibp.BF16, ibp.W8
WDT = {4: torch.int32, 2: torch.int16, 1: torch.uint8}


def build(words: np.ndarray, code: int, T: float, B: int, where: str):
    n, L = words.shape
    rows_t = to_torch(words, where)
    meta = gpu_meta(rows_t, code, T, B)
    store = GpuStore(n, L, code, B, where)
    gpu_compress(rows_t, meta, store)
    torch.cuda.synchronize()
    assert int(store.status.item()) == 0
    return store, meta


def dedup_gather(store: GpuStore, meta: torch.Tensor, idx: np.ndarray, fill: int = 0):
    n_idx = idx.size
    wdt = WDT[ibp.WIDTH[store.dtype] // 8]
    out = torch.full((n_idx, store.row_elems), fill, dtype=wdt, device="cuda")
    nbytes = ibp.gather_dedup_scratch_bytes(n_idx, store.row_elems, store.dtype, store.B)
    scratch = torch.empty((max(nbytes, 16) + 15) // 16 * 16, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ibp.decompress_gather_dedup(store.slots, store.n_rows, store.row_elems, store.dtype, store.B,
                                store.bitmask, meta, torch.from_numpy(idx).cuda(), out, scratch,
                                status)
    torch.cuda.synchronize()
    return out, int(status.item())


def full_check(words: np.ndarray, code: int, T: float, B: int, idx: np.ndarray, where: str):
    store, meta = build(words, code, T, B, where)
    out, st = dedup_gather(store, meta, idx)
    assert st == 0
    got = from_torch(out, words.dtype)
    assert np.array_equal(got, words[idx])
    plain, st2 = gpu_gather(store, meta, idx)
    assert st2 == 0 and torch.equal(plain, out)
    mask, bitval, o_slots, o_bm, _ = oracle_store(words, T, B)
    pick = np.unique(np.random.default_rng(idx.size).integers(0, idx.size, size=min(500, idx.size)))
    o_out, rc = oracle.decompress_gather(o_slots, words.shape[0], words.shape[1], words.dtype, B,
                                         o_bm, mask, bitval, idx[pick])
    assert rc == 0 and np.array_equal(got[pick], o_out)


@pytest.mark.parametrize("where", ["host", "device"])
def test_gnn_dense_zipf(where):
    """Dense GNN features, Zipf(1.0) indices: about 40% of the positions are distinct."""
    words = words_of(gen.gnn_dense(50_000))
    idx = gen.zipf_indices(words.shape[0], 30_000, 1.0, part=3, workload=gen.GNN_DENSE)
    assert np.unique(idx).size < 0.8 * idx.size
    full_check(words, FP32, 0.9, 32, idx, where)


@pytest.mark.parametrize("where", ["host", "device"])
def test_sparse_long_rows(where):
    """2 KB rows (warp-specialised kernel in HBM), uniform and repeated indices."""
    words = words_of(gen.gnn_sparse(4000))
    g = np.random.default_rng(9)
    idx = np.concatenate([g.integers(0, 4000, size=3000), np.full(500, 17)]).astype(np.int64)
    g.shuffle(idx)
    full_check(words, FP32, 0.9, 32, idx, where)


@pytest.mark.parametrize("code,np_dt,B,L", [(BF16, np.uint16, 64, 4096), (FP16, np.uint16, 32, 72),
                                            (W8, np.uint8, 64, 4112), (W8, np.uint8, 32, 48),
                                            (FP32, np.uint32, 64, 1060)])
def test_shapes(code, np_dt, B, L):
    g = np.random.default_rng(L + B)
    w = 8 * np.dtype(np_dt).itemsize
    n = 400
    base = g.integers(0, 1 << w, size=(n, L), dtype=np.uint64)
    hi = np.uint64(((1 << w) - 1) ^ ((1 << (w // 2 + 1)) - 1))
    flip = g.random(size=(n, L)) < 0.002
    words = np.where(flip, base, (base & ~hi) | (np.uint64(0x3F1E3F1E) & hi)).astype(np_dt)
    idx = g.zipf(1.3, size=1500).astype(np.int64) % n
    full_check(words, code, 0.9, B, idx, "device" if L > 1000 else "host")


def test_all_distinct_and_one_row():
    words = words_of(gen.tiny_fp32(4096))
    perm = np.random.default_rng(1).permutation(4096).astype(np.int64)
    full_check(words, FP32, 0.9, 32, perm, "device")
    full_check(words, FP32, 0.9, 32, np.full(20_000, 4095, dtype=np.int64), "host")
    full_check(words, FP32, 0.9, 32, np.array([7], dtype=np.int64), "device")


def test_few_hot_rows_across_many_blocks():
    # 50,003 positions over 40 rows: every row repeats inside each 1024-position block
    # of the hash pass and across all of them; bad indices are scattered in between
    words = words_of(gen.tiny_fp32(4096))
    g = np.random.default_rng(5)
    idx = g.integers(0, 40, size=50_003).astype(np.int64) * 97
    bad = g.choice(idx.size, size=300, replace=False)
    idx[bad[:150]] = -3
    idx[bad[150:]] = 4096
    store, meta = build(words, FP32, 0.9, 32, "device")
    out, st = dedup_gather(store, meta, idx, fill=7)
    assert st == ibp.ERR_INDEX
    got = from_torch(out, np.uint32)
    good = np.setdiff1d(np.arange(idx.size), bad)
    assert np.array_equal(got[good], words[idx[good]])
    assert np.all(got[bad] == 7)


def test_bad_indices_leave_rows_untouched():
    words = words_of(gen.tiny_fp32(1000))
    store, meta = build(words, FP32, 0.9, 32, "device")
    idx = np.array([5, -1, 5, 1000, 999, 1 << 45, 5, 0], dtype=np.int64)
    out, st = dedup_gather(store, meta, idx, fill=7)
    assert st == ibp.ERR_INDEX
    got = from_torch(out, np.uint32)
    good = [0, 2, 4, 6, 7]
    assert np.array_equal(got[good], words[idx[good]])
    assert np.all(got[[1, 3, 5]] == 7)


def test_empty_and_argument_errors():
    words = words_of(gen.tiny_fp32(64))
    store, meta = build(words, FP32, 0.9, 32, "device")
    out, st = dedup_gather(store, meta, np.zeros(0, dtype=np.int64))
    assert st == 0 and out.numel() == 0
    idx = torch.zeros(10, dtype=torch.int64, device="cuda")
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    res = torch.empty((10, 128), dtype=torch.int32, device="cuda")
    with pytest.raises(ibp.IBPError) as e:
        ibp.decompress_gather_dedup(store.slots, 64, 128, FP32, 32, store.bitmask, meta, idx, res,
                                    small)
    assert e.value.code == ibp.ERR_ARG
    with pytest.raises(ibp.IBPError) as e:
        ibp.gather_dedup_scratch_bytes(1 << 24, 128, FP32, 32)
    assert e.value.code == ibp.ERR_UNSUPPORTED
