"""Seeded random configurations through every GPU path against the oracle (needs a GPU).

Each case draws a width (8/16/32 bits), a block size, a row length (with and without
a shorter last block), a row count, a threshold and a data recipe (columns with
their own constant high bits, rare exceptions, raw rows), then checks metadata,
compression, the slotted, sized, packed and range gathers, the saving-aware mask and
per-position metadata against the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import lossless_bit_level_gb300 as ibp
import oracle
from codec_harness import GpuStore, bitmask_np, compare_slots, from_torch, gpu_compress, \
    gpu_gather, gpu_meta, row_bits_np, slots_np, to_torch

pytestmark = pytest.mark.gpu

WIDTHS = {8: (np.uint8, ibp.W8), 16: (np.uint16, ibp.BF16), 32: (np.uint32, ibp.FP32)}


def draw_case(seed: int, long_rows: bool = False):
    g = np.random.default_rng([seed, 1] if long_rows else seed)
    w = int(g.choice([8, 16, 32]))
    np_dt, code = WIDTHS[w]
    B = int(g.choice([32, 64]))
    step = 128 // w  # elements per 16 bytes: keeps shorter last blocks legal
    if long_rows:  # rows of 2 KiB + 16 bytes to 40 KiB
        L = step * int(g.integers(129, 2561))
    elif g.random() < 0.5:
        L = B * int(g.integers(1, 12))
    else:
        L = step * int(g.integers(1, 4 * B // step * 3))
        L = max(L, step)
    n = int(g.integers(1, 120 if long_rows else 700))
    T = float(g.choice([0.5, 0.8, 0.9, 0.97, 1.0]))
    colhi = np.array([((1 << w) - 1) ^ ((1 << int(k)) - 1) for k in g.integers(1, w, size=L)],
                     dtype=np.uint64)
    if g.random() < 0.5:  # one shared constant pattern instead of per-column ones
        colhi[:] = colhi[0]
    colconst = g.integers(0, 1 << w, size=L, dtype=np.uint64)
    base = g.integers(0, 1 << w, size=(n, L), dtype=np.uint64)
    flip = g.random(size=(n, L)) < float(g.choice([0.0, 0.001, 0.01, 0.1]))
    words = np.where(flip, base, (base & ~colhi) | (colconst & colhi)).astype(np_dt)
    if n > 3:  # some rows with no pattern at all (stored raw)
        k = int(g.integers(2, 9))
        words[::k] = base[::k].astype(np_dt)
    return words, code, B, T, g


@pytest.mark.parametrize("seed", range(120))
def test_random_case(seed):
    run_case(seed, *draw_case(seed))


@pytest.mark.parametrize("seed", range(40))
def test_random_long_rows(seed):
    """Rows over 2 KiB (one CTA per row up to 32 KiB, one warp per row beyond)."""
    run_case(seed, *draw_case(seed, long_rows=True))


def run_case(seed, words, code, B, T, g):
    n, L = words.shape
    raw = L * words.dtype.itemsize
    wdt = {4: torch.int32, 2: torch.int16, 1: torch.uint8}[words.dtype.itemsize]
    # threshold metadata, compression, slotted gather
    mask, bitval = oracle.build_meta(words, T)
    o_slots, o_bm, o_rb = oracle.compress(words, B, mask, bitval)
    where = "host" if seed % 3 == 0 else "device"
    rows_t = to_torch(words, where)
    meta = gpu_meta(rows_t, code, T, B)
    mv = meta.cpu().numpy().view(np.uint32)
    assert (int(mv[0]), int(mv[1])) == (mask, bitval)
    store = GpuStore(n, L, code, B, where)
    gpu_compress(rows_t, meta, store)
    torch.cuda.synchronize()
    assert np.array_equal(bitmask_np(store), o_bm)
    assert np.array_equal(row_bits_np(store), o_rb)
    compare_slots(slots_np(store), o_slots, o_bm, o_rb, raw)
    idx = g.integers(0, n, size=int(g.integers(1, 1500))).astype(np.int64)
    out, st = gpu_gather(store, meta, idx)
    assert st == 0 and np.array_equal(from_torch(out, words.dtype), words[idx])
    it = torch.from_numpy(idx).cuda()
    # sized gather
    out2 = torch.zeros_like(out)
    sts = torch.zeros(1, dtype=torch.int32, device="cuda")
    ibp.decompress_gather_sized(store.slots, n, L, code, B, store.bitmask, store.row_bits, meta,
                                it, out2, sts)
    # range
    b0 = int(g.integers(0, n))
    cnt = int(g.integers(1, n - b0 + 1))
    out3 = torch.zeros((cnt, L), dtype=wdt, device="cuda")
    ibp.decompress_range(store.slots, n, L, code, B, store.bitmask, meta, b0, cnt, out3, sts)
    # packed store of a random selection
    sel = g.integers(0, n, size=int(g.integers(1, 2 * n + 1))).astype(np.int64)
    o_off, o_packed, o_pbm, o_prb = oracle.pack(o_slots, L, words.dtype, o_bm, o_rb, sel)
    sel_t = torch.from_numpy(sel).cuda()
    offsets = torch.zeros(sel.size + 1, dtype=torch.int64, device="cuda")
    kscr = torch.empty(ibp.pack_scratch_bytes(sel.size) // 8 + 1, dtype=torch.int64,
                       device="cuda")
    ibp.pack_offsets(store.bitmask, store.row_bits, n, L, code, offsets, kscr, sel=sel_t,
                     status=sts)
    packed = torch.zeros(max(int(o_off[-1]), 16), dtype=torch.uint8, device="cuda")
    kbm = torch.zeros((sel.size + 31) // 32 + 1, dtype=torch.int32, device="cuda")
    ibp.pack(store.slots, n, L, code, store.bitmask, store.row_bits, offsets, packed, kbm,
             sel=sel_t, status=sts)
    pidx = g.integers(0, sel.size, size=500).astype(np.int64)
    out4 = torch.zeros((pidx.size, L), dtype=wdt, device="cuda")
    ibp.decompress_gather_packed(packed[: int(o_off[-1])] if int(o_off[-1]) else packed, offsets,
                                 sel.size, L, code, B, kbm, meta, torch.from_numpy(pidx).cuda(),
                                 out4, sts)
    torch.cuda.synchronize()
    assert int(sts.item()) == 0
    assert np.array_equal(from_torch(out2, words.dtype), words[idx])
    assert np.array_equal(from_torch(out3, words.dtype), words[b0:b0 + cnt])
    assert np.array_equal(offsets.cpu().numpy(), o_off)
    assert np.array_equal(from_torch(out4, words.dtype), words[sel[pidx]])
    # saving-aware metadata
    sm, sbv, cands = oracle.select_meta(words, T, B)
    smeta = torch.zeros(4, dtype=torch.int32, device="cuda")
    sscr = torch.empty(ibp.meta_select_scratch_bytes() // 4, dtype=torch.int32, device="cuda")
    cand = torch.zeros((ibp.MAX_MASK_CANDIDATES, 4), dtype=torch.int32, device="cuda")
    ibp.build_meta_select(rows_t, T, B, smeta, sscr, cand, dtype=code)
    torch.cuda.synchronize()
    assert smeta.cpu().numpy().view(np.uint32)[:2].tolist() == [sm, sbv]
    assert [(m, b) for m, _, b in ibp.read_candidates(cand)] == cands
    # per-position metadata (rows up to 16 KiB)
    if raw <= 16384:
        o_pm, o_pb = oracle.build_meta_positions(words, T)
        p_slots, p_bm, p_rb = oracle.compress_positions(words, B, o_pm, o_pb)
        pm = torch.zeros(L, dtype=torch.int32, device="cuda")
        pb = torch.zeros(L, dtype=torch.int32, device="cuda")
        pscr = torch.empty(ibp.meta_positions_scratch_bytes(L, code) // 8, dtype=torch.int64,
                           device="cuda")
        ibp.build_meta_positions(rows_t, T, B, pm, pb, pscr, dtype=code)
        pstore = GpuStore(n, L, code, B, "device")
        ibp.compress_positions(rows_t, B, pm, pb, pstore.slots, pstore.bitmask, pstore.row_bits,
                               dtype=code)
        out5 = torch.zeros_like(out)
        ibp.decompress_gather_positions(pstore.slots, n, L, code, B, pstore.bitmask, pm, pb, it,
                                        out5, sts)
        torch.cuda.synchronize()
        assert np.array_equal(pm.cpu().numpy().view(np.uint32), o_pm)
        assert np.array_equal(pb.cpu().numpy().view(np.uint32), o_pb)
        assert np.array_equal(bitmask_np(pstore), p_bm)
        assert np.array_equal(row_bits_np(pstore), p_rb)
        compare_slots(slots_np(pstore), p_slots, p_bm, p_rb, raw)
        assert int(sts.item()) == 0
        assert np.array_equal(from_torch(out5, words.dtype), words[idx])
