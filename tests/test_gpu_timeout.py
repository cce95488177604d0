"""The gather's bounded waits run out on the GPU, and the stream and the codec stay
usable afterwards.

The warp-specialised decompress-gather (slots in device memory, rows over 1 KiB)
passes work from planner warps to decoder warps through shared-memory barriers;
every wait on them is bounded ("Reducing the GPU Memory Bottleneck with Lossless
Compression for ML -- Extended", technical summary, "Core algorithm", decompression,
is the stage; the bound is this library's). The testing hooks (include/ibp_testing.h)
make the planners keep their plans to themselves -- a barrier that nothing completes
-- and lower the limit to 1 ms: the decoders' waits run out, the call must record
IBP_ERR_TIMEOUT, the stream must complete, and the next gather with the hooks cleared
on the same stream must be bit-exact against the oracle. No GPU fault, trap or endless
wait is involved: every warp gives up within the limit and returns."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ibp_inputs as gen
import lossless_bit_level_gb300 as ibp
import oracle
from codec_harness import GpuStore, gpu_compress, gpu_meta, to_torch

pytestmark = pytest.mark.gpu


def test_wait_runs_out_then_the_stream_recovers():
    words = gen.gnn_sparse().view(np.uint32)  # 500,000 x 512 FP32: 2 KiB rows
    n, L = words.shape
    T, B = 0.9, 32
    rows = to_torch(words, "device")
    meta = gpu_meta(rows, ibp.FP32, T, B)
    store = GpuStore(n, L, ibp.FP32, B, "device")
    gpu_compress(rows, meta, store)
    torch.cuda.synchronize()
    assert int(store.status.item()) == 0
    del rows
    idx = gen.uniform_indices(n, 100_000, part=11, workload=gen.GNN_SPARSE)
    it = torch.from_numpy(idx).cuda()
    out = torch.zeros((idx.size, L), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    prev = ibp.testing_set_wait_limit_ns(1_000_000)
    prev_w = ibp.testing_withhold_plans(True)
    try:
        ibp.decompress_gather(store.slots, n, L, ibp.FP32, B, store.bitmask, meta, it, out,
                              status, stream=stream)
    finally:
        ibp.testing_withhold_plans(prev_w)
        ibp.testing_set_wait_limit_ns(prev)
    stream.synchronize()  # the call ends: no wait is left without a bound
    assert int(status.item()) == ibp.ERR_TIMEOUT
    # the next gather on the same stream, with the default limit, is exact
    status.zero_()
    out.zero_()
    torch.cuda.current_stream().wait_stream(stream)
    ibp.decompress_gather(store.slots, n, L, ibp.FP32, B, store.bitmask, meta, it, out, status,
                          stream=stream)
    stream.synchronize()
    assert int(status.item()) == 0
    got = out.cpu().numpy().view(np.uint32)
    assert np.array_equal(got, words[idx])
    # and against the oracle's own gather of a sample of the rows
    mask, bitval = oracle.build_meta(words, T)
    m = meta.cpu().numpy().view(np.uint32)
    assert (int(m[0]), int(m[1])) == (mask, bitval)
    pick = np.unique(idx[:2000])
    o_slots, o_bm, _ = oracle.compress(words[pick], B, mask, bitval)
    pos = np.searchsorted(pick, idx[:2000])
    o_out, rc = oracle.decompress_gather(o_slots, pick.size, L, np.uint32, B, o_bm, mask, bitval,
                                         pos)
    assert rc == 0 and np.array_equal(got[:2000], o_out)
