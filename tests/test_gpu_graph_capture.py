"""Every compute call of the C ABI captured in one CUDA graph and replayed (needs a GPU).

The header states that the calls may be captured once their argument checks pass;
the test builds metadata (threshold, saving-aware, per-position), compresses, gathers
(plain, packed, per-position and de-duplicated, the last for short and long rows),
packs and streams a range inside one capture, replays the graph on fresh inputs and
checks every output against the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ibp_inputs as gen
import lossless_bit_level_gb300 as ibp
import oracle
from codec_harness import words_of

pytestmark = pytest.mark.gpu


def test_whole_api_in_one_graph():
    dev = torch.device("cuda")
    n, L, B, T = 3000, 128, 32, 0.9
    FP32 = ibp.FP32
    rows = torch.zeros((n, L), dtype=torch.int32, device=dev)
    meta = torch.zeros(4, dtype=torch.int32, device=dev)
    smeta = torch.zeros(4, dtype=torch.int32, device=dev)
    scr = torch.empty(ibp.meta_scratch_bytes() // 4, dtype=torch.int32, device=dev)
    sscr = torch.empty(ibp.meta_select_scratch_bytes() // 4, dtype=torch.int32, device=dev)
    cand = torch.zeros((ibp.MAX_MASK_CANDIDATES, 4), dtype=torch.int32, device=dev)
    pm = torch.zeros(L, dtype=torch.int32, device=dev)
    pb = torch.zeros(L, dtype=torch.int32, device=dev)
    pscr = torch.empty(ibp.meta_positions_scratch_bytes(L, FP32) // 8, dtype=torch.int64,
                       device=dev)
    sb = ibp.slot_bytes(L, FP32)
    slots = torch.zeros((n, sb), dtype=torch.uint8, device=dev)
    pslots = torch.zeros((n, sb), dtype=torch.uint8, device=dev)
    bm = torch.zeros(((n + 31) // 32,), dtype=torch.int32, device=dev)
    pbm = torch.zeros_like(bm)
    rb = torch.zeros(n, dtype=torch.int32, device=dev)
    prb = torch.zeros_like(rb)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    idx = torch.zeros(1000, dtype=torch.int64, device=dev)
    out = torch.zeros((1000, L), dtype=torch.int32, device=dev)
    pout = torch.zeros_like(out)
    rout = torch.zeros((n, L), dtype=torch.int32, device=dev)
    offsets = torch.zeros(n + 1, dtype=torch.int64, device=dev)
    kscr = torch.empty(ibp.pack_scratch_bytes(n) // 8 + 1, dtype=torch.int64, device=dev)
    packed = torch.zeros(n * sb, dtype=torch.uint8, device=dev)
    kbm = torch.zeros_like(bm)
    kout = torch.zeros_like(out)
    dout = torch.zeros_like(out)
    dscr = torch.empty(ibp.gather_dedup_scratch_bytes(1000, L, FP32, B), dtype=torch.uint8,
                       device=dev)
    # long rows (several gather units each): the de-duplicated gather's hash-pass path
    Ll = 2048
    lrows = torch.zeros((300, Ll), dtype=torch.int32, device=dev)
    lmeta = torch.zeros(4, dtype=torch.int32, device=dev)
    lsb = ibp.slot_bytes(Ll, FP32)
    lslots = torch.zeros((300, lsb), dtype=torch.uint8, device=dev)
    lbm = torch.zeros(((300 + 31) // 32,), dtype=torch.int32, device=dev)
    lidx = torch.zeros(500, dtype=torch.int64, device=dev)
    lout = torch.zeros((500, Ll), dtype=torch.int32, device=dev)
    lscr = torch.empty(ibp.gather_dedup_scratch_bytes(500, Ll, FP32, B), dtype=torch.uint8,
                       device=dev)

    def calls(stream):
        ibp.build_meta(rows, T, B, meta, scr, dtype=FP32, stream=stream)
        ibp.build_meta_select(rows, T, B, smeta, sscr, cand, dtype=FP32, stream=stream)
        ibp.compress(rows, B, meta, slots, bm, rb, status, dtype=FP32, stream=stream)
        ibp.decompress_gather(slots, n, L, FP32, B, bm, meta, idx, out, status, stream=stream)
        ibp.decompress_range(slots, n, L, FP32, B, bm, meta, 0, n, rout, status, stream=stream)
        ibp.pack_offsets(bm, rb, n, L, FP32, offsets, kscr, status=status, stream=stream)
        ibp.pack(slots, n, L, FP32, bm, rb, offsets, packed, kbm, status=status, stream=stream)
        ibp.decompress_gather_packed(packed, offsets, n, L, FP32, B, kbm, meta, idx, kout,
                                     status, stream=stream)
        ibp.build_meta_positions(rows, T, B, pm, pb, pscr, dtype=FP32, stream=stream)
        ibp.compress_positions(rows, B, pm, pb, pslots, pbm, prb, dtype=FP32, stream=stream)
        ibp.decompress_gather_positions(pslots, n, L, FP32, B, pbm, pm, pb, idx, pout, status,
                                        stream=stream)
        ibp.decompress_gather_dedup(slots, n, L, FP32, B, bm, meta, idx, dout, dscr, status,
                                    stream=stream)
        ibp.build_meta(lrows, T, B, lmeta, scr, dtype=FP32, stream=stream)
        ibp.compress(lrows, B, lmeta, lslots, lbm, None, status, dtype=FP32, stream=stream)
        ibp.decompress_gather_dedup(lslots, 300, Ll, FP32, B, lbm, lmeta, lidx, lout, lscr,
                                    status, stream=stream)

    s = torch.cuda.Stream()
    calls(s)  # first calls outside the capture (per-device lookups happen once)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls(s)
    for k in range(2):
        words = words_of(gen.gnn_dense(n)) if k == 0 else words_of(gen.dlrm_table(7, n))
        ix = np.random.default_rng(k).integers(0, n, size=1000)
        rows.copy_(torch.from_numpy(words.view(np.int32)))
        idx.copy_(torch.from_numpy(ix))
        lwords = words_of(gen.gnn_dense(300 * 16)).reshape(300, Ll)
        lix = np.random.default_rng(10 + k).zipf(1.2, size=500).astype(np.int64) % 300
        lrows.copy_(torch.from_numpy(lwords.view(np.int32)))
        lidx.copy_(torch.from_numpy(lix))
        status.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        mask, bitval = oracle.build_meta(words, T)
        assert meta.cpu().numpy().view(np.uint32)[:2].tolist() == [mask, bitval]
        sm, sbv, _ = oracle.select_meta(words, T, B)
        assert smeta.cpu().numpy().view(np.uint32)[:2].tolist() == [sm, sbv]
        o_pm, o_pb = oracle.build_meta_positions(words, T)
        assert np.array_equal(pm.cpu().numpy().view(np.uint32), o_pm)
        assert np.array_equal(pb.cpu().numpy().view(np.uint32), o_pb)
        for t in (out, kout, pout, dout):
            assert np.array_equal(t.cpu().numpy().view(np.uint32), words[ix])
        assert np.array_equal(lout.cpu().numpy().view(np.uint32), lwords[lix])
        assert np.array_equal(rout.cpu().numpy().view(np.uint32), words)
        _, o_bm, o_rb = oracle.compress(words, B, mask, bitval)
        assert np.array_equal(bm.cpu().numpy().view(np.uint32), o_bm)
        assert np.array_equal(rb.cpu().numpy().view(np.uint32), o_rb)
