"""Packed store (rows end to end) on the GPU against the oracle (needs a GPU).

Offsets are compared exactly, entries byte for byte over each row's used prefix,
the packed bitmask and bit counts exactly; gathers from the packed store element by
element against the oracle's gather of its own packed store and the original rows."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ibp_inputs as gen
import lossless_bit_level_gb300 as ibp
import oracle
from codec_harness import GpuStore, gpu_compress, gpu_meta, meta_tensor, oracle_store, to_torch, \
    words_of

pytestmark = pytest.mark.gpu

FP32, FP16, BF16, W8 = ibp.FP32, ibp.FP16, ibp.BF16, ibp.W8


class GpuPacked:
    """A packed store built on the GPU from a slotted GpuStore."""

    def __init__(self, store: GpuStore, sel: np.ndarray | None, where: str):
        n_sel = store.n_rows if sel is None else sel.size
        self.n = n_sel
        self.sel_t = None if sel is None else torch.from_numpy(sel.astype(np.int64)).cuda()
        self.offsets = torch.zeros(n_sel + 1, dtype=torch.int64, device="cuda")
        scratch = torch.empty(ibp.pack_scratch_bytes(n_sel) // 8 + 1, dtype=torch.int64,
                              device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        ibp.pack_offsets(store.bitmask, store.row_bits, store.n_rows, store.row_elems, store.dtype,
                         self.offsets, scratch, sel=self.sel_t, n_sel=n_sel, status=self.status)
        total = int(self.offsets[-1].item())
        if where == "device":
            self.packed = torch.zeros(max(total, 16), dtype=torch.uint8, device="cuda")
        else:
            self.packed = torch.zeros(max(total, 16), dtype=torch.uint8, pin_memory=True)
        self.packed = self.packed[:total] if total else self.packed[:16]
        self.bitmask = torch.zeros((n_sel + 31) // 32 + 1, dtype=torch.int32, device="cuda")
        self.row_bits = torch.zeros(max(n_sel, 1), dtype=torch.int32, device="cuda")
        ibp.pack(store.slots, store.n_rows, store.row_elems, store.dtype, store.bitmask,
                 store.row_bits, self.offsets, self.packed, self.bitmask, self.row_bits,
                 sel=self.sel_t, n_sel=n_sel, status=self.status)
        torch.cuda.synchronize()


def packed_gather(p: GpuPacked, L: int, dtype_code: int, B: int, meta, idx: np.ndarray):
    wdt = {32: torch.int32, 16: torch.int16, 8: torch.uint8}[ibp.WIDTH[dtype_code]]
    out = torch.zeros((idx.size, L), dtype=wdt, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ibp.decompress_gather_packed(p.packed, p.offsets, p.n, L, dtype_code, B, p.bitmask, meta,
                                 torch.from_numpy(idx.astype(np.int64)).cuda(), out, status)
    torch.cuda.synchronize()
    return out, int(status.item())


def check_packed(words, dtype_code, T, B, sel, where, rows_where="device"):
    n, L = words.shape
    mask, bitval, o_slots, o_bitmask, o_row_bits = oracle_store(words, T, B)
    o_off, o_packed, o_pbm, o_prb = oracle.pack(o_slots, L, words.dtype, o_bitmask, o_row_bits,
                                                sel)
    rows_t = to_torch(words, rows_where)
    meta = gpu_meta(rows_t, dtype_code, T, B)
    store = GpuStore(n, L, dtype_code, B, rows_where)
    gpu_compress(rows_t, meta, store)
    p = GpuPacked(store, sel, where)
    assert int(p.status.item()) == 0
    off = p.offsets.cpu().numpy()
    assert np.array_equal(off, o_off)
    n_sel = off.size - 1
    assert np.array_equal(p.bitmask.cpu().numpy().view(np.uint32)[: o_pbm.size], o_pbm)
    assert np.array_equal(p.row_bits.cpu().numpy().view(np.uint32)[:n_sel], o_prb)
    got = p.packed.cpu().numpy()
    raw = L * words.dtype.itemsize
    for i in range(n_sel):
        c = (o_pbm[i // 32] >> (i % 32)) & 1
        used = 4 * ((int(o_prb[i]) + 31) // 32) if c else raw
        assert np.array_equal(got[off[i]: off[i] + used], o_packed[off[i]: off[i] + used]), i
    g = np.random.default_rng(n_sel)
    idx = np.concatenate([g.integers(0, max(n_sel, 1), size=3 * max(n_sel, 1)),
                          [0, n_sel - 1]]).astype(np.int64) if n_sel else np.zeros(0, np.int64)
    out, st = packed_gather(p, L, dtype_code, B, meta, idx)
    assert st == 0
    o_out, rc = oracle.decompress_gather_packed(o_packed, o_off, L, words.dtype, B, o_pbm, mask,
                                                bitval, idx)
    assert rc == 0
    res = out.cpu().numpy().view(words.dtype)
    assert np.array_equal(res, o_out)
    src = np.arange(n) if sel is None else sel
    assert np.array_equal(res, words[src[idx]])
    return p, store, meta


@pytest.mark.parametrize("where", ["device", "host"])
def test_gnn_dense_cache(where):
    """A cache of 6000 hot rows (Zipf, with repeats) of a dense-GNN prefix."""
    words = words_of(gen.gnn_dense(20_000))
    sel = gen.zipf_indices(words.shape[0], 6000, 1.0, workload=gen.GNN_DENSE)
    check_packed(words, FP32, 0.9, 32, sel, where)


@pytest.mark.parametrize("where", ["device", "host"])
def test_gnn_sparse_all_rows(where):
    """Every row (no selection list): 2 KB rows, one segment, staged whole."""
    words = words_of(gen.gnn_sparse(3000))
    check_packed(words, FP32, 0.9, 32, None, where)


def test_llm_kv_multi_segment():
    """8 KB BF16 rows: two segments per row, header path with entry-length checks."""
    words = gen.llm_kv(0, 1, n_rows=600)
    sel = np.random.default_rng(1).permutation(600)[:400]
    check_packed(words, BF16, 0.9, 64, sel, "device")


def test_llm_down_rows_host():
    words = gen.llm_weight(1, "down", n_rows=120)
    check_packed(words, BF16, 0.9, 64, None, "host")


@pytest.mark.parametrize("dtype_code,np_dt,B,L", [
    (FP32, np.uint32, 32, 96), (FP16, np.uint16, 32, 224), (BF16, np.uint16, 64, 4160),
    (FP32, np.uint32, 64, 1088), (FP32, np.uint32, 32, 100), (W8, np.uint8, 32, 48),
    (W8, np.uint8, 64, 4112)])
def test_shapes(dtype_code, np_dt, B, L):
    g = np.random.default_rng(L)
    w = 8 * np.dtype(np_dt).itemsize
    n = 300
    base = g.integers(0, 1 << w, size=(n, L), dtype=np.uint64)
    hi = np.uint64(((1 << w) - 1) ^ ((1 << (w // 2 + 1)) - 1))
    flip = g.random(size=(n, L)) < 0.002
    words = np.where(flip, base, (base & ~hi) | (np.uint64(0x3F1E3F1E) & hi)).astype(np_dt)
    words[::5] = base[::5].astype(np_dt)  # rows stored raw
    sel = g.integers(0, n, size=450)
    check_packed(words, dtype_code, 0.9, B, sel, "device")


def test_empty_selection_and_single_row():
    words = words_of(gen.tiny_fp32(64))
    check_packed(words, FP32, 0.9, 32, np.array([5], dtype=np.int64), "device")
    # n_sel = 0: offsets = [0], nothing packed, nothing gathered
    mask, bitval, _, _, _ = oracle_store(words, 0.9, 32)
    rows_t = to_torch(words, "device")
    meta = gpu_meta(rows_t, FP32, 0.9, 32)
    store = GpuStore(64, 128, FP32, 32, "device")
    gpu_compress(rows_t, meta, store)
    p = GpuPacked(store, np.zeros(0, dtype=np.int64), "device")
    assert p.offsets.cpu().tolist() == [0]
    assert int(p.status.item()) == 0


def test_bad_selection_and_corrupt_offsets():
    words = words_of(gen.tiny_fp32(256))
    n, L = words.shape
    rows_t = to_torch(words, "device")
    meta = gpu_meta(rows_t, FP32, 0.9, 32)
    store = GpuStore(n, L, FP32, 32, "device")
    gpu_compress(rows_t, meta, store)
    # a selection outside the store: index error, a 0-byte entry
    sel = np.array([3, n, 7], dtype=np.int64)
    p = GpuPacked(store, sel, "device")
    assert int(p.status.item()) == ibp.ERR_INDEX
    off = p.offsets.cpu().numpy()
    assert off[2] == off[1]
    good = GpuPacked(store, np.arange(40, dtype=np.int64), "device")
    assert int(good.status.item()) == 0
    sentinel = 0x5A5A5A5A
    for what in ("unaligned", "past_end", "short", "decreasing"):
        bad_off = good.offsets.clone()
        k = 9
        if what == "unaligned":
            bad_off[k] += 4
        elif what == "past_end":
            bad_off[k + 1] = good.packed.numel() + 16
        elif what == "short":
            bad_off[k + 1] = bad_off[k] + 16
        else:
            bad_off[k + 1] = bad_off[k] - 16
        bp = GpuPacked.__new__(GpuPacked)
        bp.__dict__.update(good.__dict__)
        bp.offsets = bad_off
        out = torch.full((3, L), sentinel, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        idx = torch.tensor([k, 2, k], dtype=torch.int64, device="cuda")
        ibp.decompress_gather_packed(bp.packed, bp.offsets, bp.n, L, FP32, 32, bp.bitmask, meta,
                                     idx, out, status)
        torch.cuda.synchronize()
        assert int(status.item()) == ibp.ERR_CORRUPT, what
        res = out.cpu().numpy().view(np.uint32)
        assert np.all(res[0] == sentinel) and np.all(res[2] == sentinel), what
        assert np.array_equal(res[1], words[2]), what


def test_packed_capacity_gain_matches_oracle_sizes():
    """The packed store of a whole dense-GNN prefix is the sum of 16-byte-rounded
    stored sizes; with the saving-aware mask the cache holds more rows per byte."""
    words = words_of(gen.gnn_dense(8000))
    n, L = words.shape
    o_mask, o_bitval, _ = oracle.select_meta(words, 0.9, 32)
    slots, bm, rb = oracle.compress(words, 32, o_mask, o_bitval)
    o_off, _, _, _ = oracle.pack(slots, L, words.dtype, bm, rb, None)
    rows_t = to_torch(words, "device")
    meta = meta_tensor(o_mask, o_bitval, FP32, 32)
    store = GpuStore(n, L, FP32, 32, "device")
    gpu_compress(rows_t, meta, store)
    p = GpuPacked(store, None, "device")
    assert np.array_equal(p.offsets.cpu().numpy(), o_off)
    assert o_off[-1] < n * L * 4
