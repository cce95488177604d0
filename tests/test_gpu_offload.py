"""Contiguous-range decompression and the overlapped offload pipeline (needs a GPU).

The range call is compared with the oracle's gather of the same rows; the pipeline's
buffers, copied out by a deliberately slow consumer, must hold every layer's original
tensors exactly (a buffer reused before its consumer finished would show up as a
mismatch)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ibp_inputs as gen
import lossless_bit_level_gb300 as ibp
import oracle
from codec_harness import GpuStore, gpu_compress, gpu_meta, oracle_store, to_torch, words_of
from lossless_bit_level_gb300.offload import CompressedTensor, OffloadPipeline, raw_loader

pytestmark = pytest.mark.gpu

FP32, BF16 = ibp.FP32, ibp.BF16


@pytest.mark.parametrize("where", ["device", "host"])
@pytest.mark.parametrize("name,dtype_code,B", [("dense", FP32, 32), ("kv", BF16, 64),
                                               ("down", BF16, 64)])
def test_decompress_range(where, name, dtype_code, B):
    words = {"dense": lambda: words_of(gen.gnn_dense(3000)),
             "kv": lambda: gen.llm_kv(3, 0, n_rows=700),
             "down": lambda: gen.llm_weight(2, "down", n_rows=96)}[name]()
    n, L = words.shape
    mask, bitval, o_slots, o_bitmask, _ = oracle_store(words, 0.9, B)
    rows_t = to_torch(words, where)
    meta = gpu_meta(rows_t, dtype_code, 0.9, B)
    store = GpuStore(n, L, dtype_code, B, where)
    gpu_compress(rows_t, meta, store)
    wdt = torch.int32 if dtype_code == FP32 else torch.int16
    for begin, count in ((0, n), (1, n - 1), (n // 3, n // 5), (n - 1, 1)):
        out = torch.zeros((count, L), dtype=wdt, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        ibp.decompress_range(store.slots, n, L, dtype_code, B, store.bitmask, meta, begin, count,
                             out, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = out.cpu().numpy().view(words.dtype)
        o_out, rc = oracle.decompress_gather(o_slots, n, L, words.dtype, B, o_bitmask, mask,
                                             bitval, np.arange(begin, begin + count))
        assert rc == 0
        assert np.array_equal(got, o_out)
        assert np.array_equal(got, words[begin:begin + count])
    with pytest.raises(ibp.IBPError):
        ibp.decompress_range(store.slots, n, L, dtype_code, B, store.bitmask, meta, n - 2, 3,
                             torch.zeros((3, L), dtype=wdt, device="cuda"))


def small_layers(n_layers: int):
    """Layers of two BF16 weight-like tensors (row counts differ, so a mix-up of
    buffers would fail), compressed into host slots."""
    dev = torch.device("cuda")
    layers, originals = [], []
    for l in range(n_layers):
        a = gen.llm_weight(l, "q", n_rows=192)[:, :512].copy()
        b = gen.llm_weight(l, "down", n_rows=64)[:, :1024].copy()
        originals.append([a, b])
        layers.append([CompressedTensor.from_words(x, BF16, 0.9, 64, dev) for x in (a, b)])
    return layers, originals


@pytest.mark.parametrize("overlap", [True, False])
@pytest.mark.parametrize("loader", ["ibp", "raw"])
def test_pipeline_delivers_every_layer(overlap, loader):
    dev = torch.device("cuda")
    layers, originals = small_layers(3)
    load = None
    if loader == "raw":
        raw = {}
        for lay, orig in zip(layers, originals):
            for t, x in zip(lay, orig):
                h = torch.empty(x.shape, dtype=torch.int16, pin_memory=True)
                h.copy_(torch.from_numpy(x.view(np.int16)))
                raw[id(t)] = h
        load = raw_loader(raw)
    pipe = OffloadPipeline(layers, dev, load=load, overlap=overlap)
    seen = []

    def consume(layer, bufs):
        torch.cuda._sleep(200_000)  # a slow consumer: reuse too early would be caught
        seen.append((layer, [b.clone() for b in bufs]))

    order = [0, 1, 2, 1, 0, 2, 2, 0]
    pipe.run(len(order), consume, order=order)
    pipe.run(3, consume, order=[2, 2, 1])  # a second run reuses the buffers at once
    pipe.synchronize()
    assert [l for l, _ in seen] == order + [2, 2, 1]
    for layer, bufs in seen:
        for got, want in zip(bufs, originals[layer]):
            assert np.array_equal(got.cpu().numpy().view(np.uint16), want)
    for lay in layers:
        for t in lay:
            assert int(t.status.item()) == 0


def test_compressed_tensor_saving_aware():
    dev = torch.device("cuda")
    x = words_of(gen.gnn_dense(4000))
    t = CompressedTensor.from_words(x, FP32, 0.9, 32, dev, saving_aware=True)
    m, bv, _ = oracle.select_meta(x, 0.9, 32)
    assert t.meta.cpu().numpy().view(np.uint32)[:2].tolist() == [m, bv]
    out = t.empty_like(dev)
    t.decompress_into(out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.uint32), x)
    assert t.stored_bytes() < t.raw_bytes
