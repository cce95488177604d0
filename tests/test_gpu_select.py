"""Saving-aware mask selection on the GPU against the oracle (needs a GPU).

Every case compares the whole candidate table (masks, bitvals, scores) and the
chosen metadata with the oracle's selection on the same rows, then checks that
compressing with the chosen metadata stores exactly the bytes its score says and
round-trips through the gather."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ibp_inputs as gen
import lossless_bit_level_gb300 as ibp
import oracle
import pins
from codec_harness import GpuStore, gpu_compress, gpu_gather, meta_values, to_torch, words_of

pytestmark = pytest.mark.gpu

FP32, FP16, BF16, W8 = ibp.FP32, ibp.FP16, ibp.BF16, ibp.W8


def gpu_select(rows_t: torch.Tensor, dtype_code: int, T: float, B: int):
    meta = torch.zeros((4,), dtype=torch.int32, device="cuda")
    scratch = torch.empty((ibp.meta_select_scratch_bytes() // 4,), dtype=torch.int32,
                          device="cuda")
    cand = torch.zeros((ibp.MAX_MASK_CANDIDATES, 4), dtype=torch.int32, device="cuda")
    ibp.build_meta_select(rows_t, T, B, meta, scratch, cand, dtype=dtype_code)
    torch.cuda.synchronize()
    return meta, ibp.read_candidates(cand)


def select_check(words: np.ndarray, dtype_code: int, T: float, B: int, where: str = "device"):
    n, L = words.shape
    o_mask, o_bitval, o_cands = oracle.select_meta(words, T, B)
    rows_t = to_torch(words, where)
    meta, cands = gpu_select(rows_t, dtype_code, T, B)
    assert meta_values(meta) == (o_mask, o_bitval, dtype_code, B)
    M0_bitval = oracle.build_meta(words, T)[1]
    assert cands == [(m, M0_bitval & m, b) for m, b in o_cands]
    # the chosen metadata stores exactly its score and round-trips
    store = GpuStore(n, L, dtype_code, B, "device")
    gpu_compress(rows_t, meta, store)
    st = ibp.query(store.bitmask, store.row_bits, n, L, dtype_code)
    assert st.stored_bytes == dict(o_cands)[o_mask]
    idx = np.random.default_rng(n).integers(0, n, size=min(2000, 4 * n)).astype(np.int64)
    out, rc = gpu_gather(store, meta, idx)
    assert rc == 0
    assert np.array_equal(out.cpu().numpy().view(words.dtype), words[idx])
    return o_mask, o_cands


def test_bit26_example():
    """The hand-worked FP32 example: the threshold mask saves nothing, dropping the
    position with one exception per row saves 88 of every 128 bytes."""
    words = pins.fp32_bit26_rows()
    mask, cands = select_check(words, FP32, 0.9, 32)
    assert mask == 0xFBFFFF00
    assert cands == [(0xFFFFFF00, 1024), (0xFBFFFF00, 320), (0x00000000, 1024)]


@pytest.mark.parametrize("name", ["tiny", "dense", "sparse", "dlrm", "w_q", "w_down", "kv"])
def test_workload_prefixes(name):
    x, dt, T, B, where = {
        "tiny": (lambda: gen.tiny_fp32(), FP32, 0.9, 32, "device"),
        "dense": (lambda: gen.gnn_dense(20_000), FP32, 0.9, 32, "host"),
        "sparse": (lambda: gen.gnn_sparse(2000), FP32, 0.9, 32, "device"),
        "dlrm": (lambda: gen.dlrm_table(1, 20_000), FP32, 0.95, 32, "host"),
        "w_q": (lambda: gen.llm_weight(0, "q", 256), BF16, 0.9, 64, "device"),
        "w_down": (lambda: gen.llm_weight(1, "down", 64), BF16, 0.9, 64, "host"),
        "kv": (lambda: gen.llm_kv(0, 0, n_rows=512), BF16, 0.9, 64, "device"),
    }[name]
    select_check(words_of(x()), dt, T, B, where)


@pytest.mark.parametrize("T", [0.0, 0.5, 0.75, 0.9, 1.0])
@pytest.mark.parametrize("dtype_code,np_dt,B,L", [
    (FP32, np.uint32, 32, 96), (FP32, np.uint32, 64, 1088), (FP16, np.uint16, 32, 224),
    (BF16, np.uint16, 64, 64), (FP16, np.uint16, 32, 32),
    (FP32, np.uint32, 32, 100), (BF16, np.uint16, 64, 4104), (W8, np.uint8, 32, 48),
    (W8, np.uint8, 64, 256), (W8, np.uint8, 32, 4112)])
def test_shapes_and_thresholds(T, dtype_code, np_dt, B, L):
    """Partial last chunk (96, 224 and 1088 words are not multiples of 128), one-block
    rows, many thresholds; exceptions in a high position spread one per block."""
    g = np.random.default_rng(L + int(100 * T))
    w = 8 * np.dtype(np_dt).itemsize
    n = 257
    base = g.integers(0, 1 << w, size=(n, L), dtype=np.uint64)
    hi = np.uint64(((1 << w) - 1) ^ ((1 << (w // 2)) - 1))
    flip = g.random(size=(n, L)) < 0.002
    words = np.where(flip, base, (base & ~hi) | (np.uint64(0x3C1E3C1E) & hi)).astype(np_dt)
    words[:, ::B] ^= np_dt(1 << (w - 4))  # one exception per block in bit w-4
    select_check(words, dtype_code, T, B)


def test_all_positions_distinct_counts():
    """T = 0 keeps all 32 positions; bit j is set in exactly j of 64 elements, so the
    32 counts are distinct and there are 33 candidates (the last scored without a
    lane of its own)."""
    e = np.arange(64, dtype=np.uint64)
    words = np.zeros(64, dtype=np.uint64)
    for j in range(32):
        words |= np.where(e < j, np.uint64(1 << j), np.uint64(0))
    words = words.astype(np.uint32).reshape(2, 32)
    mask, cands = select_check(words, FP32, 0.0, 32)
    assert len(cands) == 33


@pytest.mark.parametrize("kind", ["identical", "random", "one_row"])
def test_degenerate_inputs(kind):
    g = np.random.default_rng(3)
    if kind == "identical":
        words = np.full((100, 128), 0x3F800000, dtype=np.uint32)  # full mask, 2 candidates
    elif kind == "random":
        words = g.integers(0, 1 << 32, size=(300, 128), dtype=np.uint64).astype(np.uint32)
    else:
        words = g.integers(0, 1 << 8, size=(1, 256), dtype=np.uint64).astype(np.uint32)
    select_check(words, FP32, 0.9, 32)
