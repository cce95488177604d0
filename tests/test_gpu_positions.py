"""Per-position metadata on the GPU against the oracle (needs a GPU).

Metadata arrays, bitmask, row bits and the used prefix of every slot are compared
exactly with the oracle's; gathers element by element with the oracle's gather and
with the original rows."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ibp_inputs as gen
import lossless_bit_level_gb300 as ibp
import oracle
import pins
from codec_harness import bitmask_np, compare_slots, from_torch, row_bits_np, slots_np, to_torch, \
    words_of

pytestmark = pytest.mark.gpu

FP32, FP16, BF16, W8 = ibp.FP32, ibp.FP16, ibp.BF16, ibp.W8


def gpu_positions(words: np.ndarray, dtype_code: int, T: float, B: int, where: str = "device",
                  block_positions: bool = False):
    n, L = words.shape
    rows_t = to_torch(words, where)
    pm = torch.zeros(L, dtype=torch.int32, device="cuda")
    pb = torch.zeros(L, dtype=torch.int32, device="cuda")
    scratch = torch.empty(ibp.meta_positions_scratch_bytes(L, dtype_code) // 8, dtype=torch.int64,
                          device="cuda")
    build = ibp.build_meta_block_positions if block_positions else ibp.build_meta_positions
    build(rows_t, T, B, pm, pb, scratch, dtype=dtype_code)
    sb = ibp.slot_bytes(L, dtype_code)
    if where == "device":
        slots = torch.zeros((n, sb), dtype=torch.uint8, device="cuda")
    else:
        slots = torch.zeros((n, sb), dtype=torch.uint8, pin_memory=True)
    bitmask = torch.zeros(((n + 31) // 32,), dtype=torch.int32, device="cuda")
    row_bits = torch.zeros((n,), dtype=torch.int32, device="cuda")
    ibp.compress_positions(rows_t, B, pm, pb, slots, bitmask, row_bits, dtype=dtype_code)
    torch.cuda.synchronize()
    return pm, pb, slots, bitmask, row_bits


def check(words: np.ndarray, dtype_code: int, T: float, B: int, where: str = "device",
          block_positions: bool = False):
    n, L = words.shape
    if block_positions:
        o_pm, o_pb = oracle.build_meta_block_positions(words, T, B)
    else:
        o_pm, o_pb = oracle.build_meta_positions(words, T)
    o_slots, o_bm, o_rb = oracle.compress_positions(words, B, o_pm, o_pb)
    pm, pb, slots, bitmask, row_bits = gpu_positions(words, dtype_code, T, B, where,
                                                     block_positions)
    assert np.array_equal(pm.cpu().numpy().view(np.uint32), o_pm)
    assert np.array_equal(pb.cpu().numpy().view(np.uint32), o_pb)
    gbm = bitmask.cpu().numpy().view(np.uint32)
    grb = row_bits.cpu().numpy().view(np.uint32)
    assert np.array_equal(gbm, o_bm)
    assert np.array_equal(grb, o_rb)
    compare_slots(slots.cpu().numpy(), o_slots, o_bm, o_rb, L * words.dtype.itemsize)
    g = np.random.default_rng(L + n)
    idx = np.concatenate([g.integers(0, n, size=min(3000, 4 * n)), [0, n - 1]]).astype(np.int64)
    wdt = {4: torch.int32, 2: torch.int16, 1: torch.uint8}[words.dtype.itemsize]
    out = torch.zeros((idx.size, L), dtype=wdt, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ibp.decompress_gather_positions(slots, n, L, dtype_code, B, bitmask, pm, pb,
                                    torch.from_numpy(idx).cuda(), out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = from_torch(out, words.dtype)
    o_out, rc = oracle.decompress_gather_positions(o_slots, n, L, words.dtype, B, o_bm, o_pm,
                                                   o_pb, idx)
    assert rc == 0
    assert np.array_equal(got, o_out)
    assert np.array_equal(got, words[idx])
    return o_bm, o_rb


@pytest.mark.parametrize("where", ["device", "host"])
def test_gnn_dense_columns(where):
    """Per-column distributions: the rows' columns have their own scales."""
    check(words_of(gen.gnn_dense(20_000)), FP32, 0.99, 32, where)


@pytest.mark.parametrize("name,dt,T,B", [("sparse", FP32, 0.9, 32), ("dlrm", FP32, 0.95, 32),
                                          ("kv", BF16, 0.9, 64), ("w_q", BF16, 0.9, 64),
                                          ("tiny", FP32, 0.9, 32)])
def test_workload_prefixes(name, dt, T, B):
    x = {"sparse": lambda: gen.gnn_sparse(2000), "dlrm": lambda: gen.dlrm_table(4, 20_000),
         "kv": lambda: gen.llm_kv(1, 0, n_rows=800), "w_q": lambda: gen.llm_weight(2, "q", 200),
         "tiny": lambda: gen.tiny_fp32()}[name]()
    check(words_of(x), dt, T, B)


@pytest.mark.parametrize("dtype_code,np_dt,B,L", [
    (FP32, np.uint32, 32, 96), (FP32, np.uint32, 64, 1060), (FP16, np.uint16, 32, 72),
    (BF16, np.uint16, 64, 4104), (W8, np.uint8, 32, 48), (W8, np.uint8, 64, 4112),
    (FP32, np.uint32, 32, 4), (BF16, np.uint16, 64, 8192)])
@pytest.mark.parametrize("T", [0.75, 1.0])
def test_shapes_columns_and_tails(dtype_code, np_dt, B, L, T):
    """Columns with their own constant high bits (a different number per column),
    rare exceptions, shorter last blocks, 8-bit words, the 16 KiB row limit."""
    g = np.random.default_rng(L * 3 + int(T * 10))
    w = 8 * np.dtype(np_dt).itemsize
    n = 300
    colconst = g.integers(0, 1 << w, size=L, dtype=np.uint64)
    colhi = np.array([((1 << w) - 1) ^ ((1 << int(k)) - 1) for k in g.integers(1, w, size=L)],
                     dtype=np.uint64)
    base = g.integers(0, 1 << w, size=(n, L), dtype=np.uint64)
    flip = g.random(size=(n, L)) < 0.001
    words = np.where(flip, base, (base & ~colhi) | (colconst & colhi)).astype(np_dt)
    words[::9] = base[::9].astype(np_dt)  # rows stored raw
    check(words, dtype_code, T, B)


def test_hand_example_rows_on_gpu():
    """The hand-worked positions example, widened to GPU block sizes: the 8-byte
    pattern repeated to 64 positions, B = 32."""
    d = pins.load_hand_example("positions_example_u8.txt", np.uint8)
    words = np.tile(d["rows"], (8, 8))  # 32 rows x 64 positions
    bm, rb = check(words, W8, 1.0, 32)
    assert np.all(rb == 2 + 2 * 8 * 12)  # two blocks of 32 positions: 8 groups of 2+0+2+8 bits


def test_special_values():
    g = np.random.default_rng(5)
    for w, dt, code in ((32, np.uint32, FP32), (16, np.uint16, FP16), (8, np.uint8, W8)):
        sp = np.array(pins.special_words(w), dtype=dt)
        n, L = 200, 64
        words = sp[g.integers(0, sp.size, size=(n, L))]
        col = sp[g.integers(0, sp.size, size=L)]
        words[: n // 2] = np.where(g.random(size=(n // 2, L)) < 0.97, col[None, :],
                                   words[: n // 2])
        check(words, code, 0.9, 32)


def test_bad_index_and_row_limit():
    words = words_of(gen.tiny_fp32(256))
    n, L = words.shape
    pm, pb, slots, bitmask, row_bits = gpu_positions(words, FP32, 0.9, 32)
    out = torch.full((3, L), 7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ibp.decompress_gather_positions(slots, n, L, FP32, 32, bitmask, pm, pb,
                                    torch.tensor([1, n, 2], dtype=torch.int64, device="cuda"), out,
                                    status)
    torch.cuda.synchronize()
    assert int(status.item()) == ibp.ERR_INDEX
    res = out.cpu().numpy().view(np.uint32)
    assert np.array_equal(res[0], words[1]) and np.all(res[1] == 7)
    big = torch.zeros((4, 8200), dtype=torch.int16, device="cuda")
    with pytest.raises(ibp.IBPError) as e:
        ibp.compress_positions(big, 64, pm, pb, torch.zeros((4, 16400), dtype=torch.uint8,
                                                            device="cuda"), bitmask, dtype=BF16)
    assert e.value.code == ibp.ERR_UNSUPPORTED


@pytest.mark.parametrize("dtype_code,np_dt,B,L", [
    (FP32, np.uint32, 32, 96), (FP32, np.uint32, 64, 1060), (FP16, np.uint16, 32, 72),
    (BF16, np.uint16, 64, 4104), (W8, np.uint8, 32, 48), (W8, np.uint8, 64, 4112),
    (FP32, np.uint32, 32, 4), (BF16, np.uint16, 64, 8192)])
@pytest.mark.parametrize("T", [0.75, 0.97])
def test_block_positions_shapes_and_tails(dtype_code, np_dt, B, L, T):
    """Block-position metadata: each position within a block has its own constant
    high bits (the same in every block), rare exceptions, rows stored raw, shorter
    last blocks (whose positions are counted only where they exist), 8-bit words."""
    g = np.random.default_rng(L * 5 + int(T * 100))
    w = 8 * np.dtype(np_dt).itemsize
    n = 300
    q_of = np.arange(L) % B
    colconst = g.integers(0, 1 << w, size=B, dtype=np.uint64)[q_of]
    colhi = np.array([((1 << w) - 1) ^ ((1 << int(k)) - 1) for k in g.integers(1, w, size=B)],
                     dtype=np.uint64)[q_of]
    base = g.integers(0, 1 << w, size=(n, L), dtype=np.uint64)
    flip = g.random(size=(n, L)) < 0.01
    words = np.where(flip, base, (base & ~colhi) | (colconst & colhi)).astype(np_dt)
    words[::11] = base[::11].astype(np_dt)
    check(words, dtype_code, T, B, block_positions=True)


@pytest.mark.parametrize("where", ["device", "host"])
@pytest.mark.parametrize("name,dt,T,B", [("kv", BF16, 0.9, 64), ("dlrm", FP32, 0.95, 32),
                                          ("sparse", FP32, 0.9, 32)])
def test_block_positions_workloads(where, name, dt, T, B):
    x = {"sparse": lambda: gen.gnn_sparse(1500), "dlrm": lambda: gen.dlrm_table(3, 20_000),
         "kv": lambda: gen.llm_kv(0, 1, n_rows=600)}[name]()
    check(words_of(x), dt, T, B, where, block_positions=True)


def test_block_positions_equal_positions_for_one_block_rows():
    """With one block per row the block positions are the element positions."""
    words = words_of(gen.dlrm_table(1, 5000, row_elems=32))
    a = gpu_positions(words, FP32, 0.9, 32, block_positions=True)
    b = gpu_positions(words, FP32, 0.9, 32)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
