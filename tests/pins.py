"""Checks that pin the oracle to facts other than itself.

Each check takes an ``oracle.Oracle`` instance and raises AssertionError on a
mismatch, so the same checks run against the real oracle and against copies of it
with a mistake planted on purpose (tests/test_oracle_pins.py).

What pins what (method: "Reducing the GPU Memory Bottleneck with Lossless
Compression for ML -- Extended", technical summary, core algorithm):
  * hand-worked example (tests/golden/hand_example_fp16.txt): exact mask, bitval,
    sizes, bitmask and stream words worked out by hand;
  * brute-force meta: per-bit counts taken with numpy.unpackbits over every input
    of a small alphabet, against the preprocessing rule (majority value held by at
    least a fraction T of the sample);
  * closed forms of the preprocessing rule: T = 1 gives mask = ~(OR ^ AND),
    bitval = AND & mask; identical elements give a full mask; a tie picks 0;
  * the size formula sum_b (1 + B*(w - popcount(mask))) for matching blocks and
    (1 + B*w) otherwise, with matches found by a vectorised numpy comparison, and
    the store-compressed rule 4*ceil(bits/32) < raw bytes;
  * the stream layout rebuilt as a Python string of '0'/'1' characters;
  * lossless round trip (the decoded row equals the original word for word) on
    +-0, denormals, +-Inf, NaN payloads and all-ones words;
  * decode of the hand-worked stream words (typed in from the golden file, not
    produced by the oracle);
  * 8-bit words and rows ending in a shorter block: a hand-worked example
    (tests/golden/hand_example_u8_tail.txt) and the size formula with tails;
  * per-position metadata: a hand-worked example (tests/golden/positions_example_u8.txt),
    the rule checked column by column against the brute-force count, sizes with
    per-element field widths, and equal masks reproducing the shared-mask stream;
  * saving-aware mask selection: two hand-worked examples
    (tests/golden/select_examples.txt) and a threshold sweep (every distinct mask
    the threshold rule gives for thresholds at or above T, plus the empty mask,
    scored with the numpy size formula) that must reach the same minimum;
  * packed store: the hand-worked rows packed in a chosen order (entry sizes and
    bytes typed in from the golden file), offsets from the size formula on random
    stores, lossless gathers from the packed bytes, and a truncated entry reported
    as corrupt.
"""
from __future__ import annotations

import itertools
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_hand_example(name: str = "hand_example_fp16.txt", dtype=np.uint16):
    rows, streams = [], []
    d = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "row":
                rows.append([int(v, 16) for v in vals])
            elif key == "stream":
                streams.append([int(v, 16) for v in vals])
            elif key in ("mask", "bitval", "bitmask"):
                d[key] = int(vals[0], 16)
            elif key == "row_bits":
                d[key] = [int(v) for v in vals]
            elif key == "T":
                d[key] = float(vals[0])
            elif key == "block":
                d[key] = int(vals[0])
            elif key in ("pmask", "pbitval"):
                d[key] = [int(v, 16) for v in vals]
    d["rows"] = np.array(rows, dtype=dtype)
    d["streams"] = streams
    return d


def wmask(w):
    return (1 << w) - 1


def bits_of(words: np.ndarray) -> np.ndarray:
    """[..., w] array of bits (bit j of each little-endian word) via unpackbits."""
    a = np.ascontiguousarray(words)
    w = 8 * a.dtype.itemsize
    b = np.unpackbits(a.view(np.uint8).reshape(a.shape + (w // 8,)), axis=-1, bitorder="little")
    return b.reshape(a.shape + (w,))


def brute_meta(words: np.ndarray, T: float):
    flat = np.ascontiguousarray(words).reshape(-1)
    w = 8 * flat.dtype.itemsize
    n = flat.size
    ones = bits_of(flat).sum(axis=0).astype(np.int64)
    mask = bitval = 0
    for j in range(w):
        c1 = int(ones[j])
        c0 = n - c1
        v = 1 if c1 > c0 else 0
        if float(c1 if v else c0) >= T * float(n):
            mask |= 1 << j
            bitval |= v << j
    return mask, bitval


def check_hand_example(o):
    d = load_hand_example()
    mask, bitval = o.build_meta(d["rows"], d["T"])
    assert (mask, bitval) == (d["mask"], d["bitval"]), (hex(mask), hex(bitval))
    slots, bitmask, row_bits = o.compress(d["rows"], d["block"], mask, bitval)
    assert list(row_bits) == d["row_bits"], list(row_bits)
    assert int(bitmask[0]) == d["bitmask"], hex(int(bitmask[0]))
    for r, words in enumerate(d["streams"]):
        got = slots[r, : 4 * len(words)].view("<u4").tolist()
        assert got == words, (r, [hex(x) for x in got])


def check_hand_decode(o):
    """Decode slots typed in from the golden file (not produced by the oracle)."""
    d = load_hand_example()
    n, L = d["rows"].shape
    slots = np.zeros((n, 16), dtype=np.uint8)
    for r, words in enumerate(d["streams"]):
        slots[r, : 4 * len(words)] = np.array(words, dtype="<u4").view(np.uint8)
    bitmask = np.array([d["bitmask"]], dtype=np.uint32)
    idx = np.array([1, 0, 1], dtype=np.int64)
    out, rc = o.decompress_gather(slots, n, L, np.uint16, d["block"], bitmask, d["mask"],
                                  d["bitval"], idx)
    assert rc == 0
    assert np.array_equal(out, d["rows"][idx])


FP16_ALPHABET = [0x0000, 0x8000, 0x3C00, 0xFFFF, 0x0001, 0x7C00, 0x7E01, 0x03FF]


def check_meta_exhaustive(o):
    """Every 2x2 FP16 input over an 8-word alphabet (+-0, 1.0, all-ones, smallest
    denormal, +Inf, a NaN with payload, largest denormal), at several T."""
    combos = np.array(list(itertools.product(FP16_ALPHABET, repeat=4)), dtype=np.uint16)
    for T in (0.0, 0.5, 0.75, 0.9, 1.0):
        for c in combos:
            got = o.build_meta(c.reshape(2, 2), T)
            exp = brute_meta(c, T)
            assert got == exp, (c, T, got, exp)


def check_meta_closed_forms(o):
    g = np.random.default_rng(12345)
    for dt, w in ((np.uint32, 32), (np.uint16, 16)):
        for trial in range(20):
            n = int(g.integers(1, 200))
            x = g.integers(0, 1 << w, size=n, dtype=np.uint64).astype(dt)
            # force some bits constant so T = 1 has something to find
            keep = int(g.integers(0, 1 << w))
            fixed = int(g.integers(0, 1 << w))
            x = ((x.astype(np.uint64) & ~np.uint64(keep)) | np.uint64(fixed & keep)).astype(dt)
            OR = int(np.bitwise_or.reduce(x.astype(np.uint64)))
            AND = int(np.bitwise_and.reduce(x.astype(np.uint64)))
            mask, bitval = o.build_meta(x, 1.0)
            exp_mask = ~(OR ^ AND) & wmask(w)
            assert mask == exp_mask, (hex(mask), hex(exp_mask))
            assert bitval == AND & exp_mask
            # identical elements: every position is invariant
            y = np.full(n, x[0], dtype=dt)
            assert o.build_meta(y, float(g.random())) == (wmask(w), int(x[0]))
        # a tie (one element with all bits 0, one with all bits 1) picks value 0
        t = np.array([0, wmask(w)], dtype=dt)
        assert o.build_meta(t, 0.5) == (wmask(w), 0)
        assert o.build_meta(t, 0.51) == (0, 0)
    # threshold boundary: 9 of 10 elements share bit 0 -> invariant at T = 0.9,
    # 8 of 10 -> not
    a = np.array([1] * 9 + [0], dtype=np.uint32)
    m, b = o.build_meta(a, 0.9)
    assert m & 1 and b & 1
    a = np.array([1] * 8 + [0] * 2, dtype=np.uint32)
    m, _ = o.build_meta(a, 0.9)
    assert not (m & 1)


def block_matches(rows: np.ndarray, B: int, mask: int, bitval: int) -> np.ndarray:
    n, L = rows.shape
    wide = rows.astype(np.uint64)
    ok = (wide & np.uint64(mask)) == np.uint64(bitval)
    return ok.reshape(n, L // B, B).all(axis=2)


def row_bits_formula(rows: np.ndarray, B: int, mask: int, bitval: int) -> np.ndarray:
    """Per-row bit counts from the size formula, blocks of B elements and a shorter
    last block when the row length is not a multiple of B; matches by numpy."""
    n, L = rows.shape
    w = 8 * rows.dtype.itemsize
    m = w - bin(mask).count("1")
    ok = (rows.astype(np.uint64) & np.uint64(mask)) == np.uint64(bitval)
    bits = np.zeros(n, dtype=np.int64)
    for b0 in range(0, L, B):
        ln = min(B, L - b0)
        match = ok[:, b0:b0 + ln].all(axis=1)
        bits += 1 + np.where(match, ln * m, ln * w)
    return bits


def check_hand_example_u8_tail(o):
    """8-bit words and a two-element last block, worked by hand (golden file)."""
    d = load_hand_example("hand_example_u8_tail.txt", np.uint8)
    mask, bitval = o.build_meta(d["rows"], d["T"])
    assert (mask, bitval) == (d["mask"], d["bitval"]), (hex(mask), hex(bitval))
    slots, bitmask, row_bits = o.compress(d["rows"], d["block"], mask, bitval)
    assert list(row_bits) == d["row_bits"], list(row_bits)
    assert int(bitmask[0]) == d["bitmask"]
    assert slots[0, :4].view("<u4").tolist() == d["streams"][0]
    assert np.array_equal(slots[1, :6], d["rows"][1])  # stored raw
    # decode the typed-in stream
    typed = np.zeros_like(slots)
    typed[0, :4] = np.array(d["streams"][0], dtype="<u4").view(np.uint8)
    typed[1, :6] = d["rows"][1]
    out, rc = o.decompress_gather(typed, 2, 6, np.uint8, d["block"], bitmask, d["mask"],
                                  d["bitval"], np.array([1, 0, 0]))
    assert rc == 0 and np.array_equal(out, d["rows"][[1, 0, 0]])


def check_tail_blocks_and_bytes(o):
    """Rows whose length is not a multiple of B, for 8-, 16- and 32-bit words: bit
    counts from the formula, the store rule, and lossless round trips."""
    g = np.random.default_rng(31337)
    for dt, w, B, L in ((np.uint8, 8, 32, 80), (np.uint8, 8, 64, 100), (np.uint16, 16, 32, 40),
                        (np.uint32, 32, 64, 72), (np.uint32, 32, 5, 13), (np.uint8, 8, 3, 7),
                        (np.uint16, 16, 64, 64 + 1)):
        n = 48
        base = g.integers(0, 1 << w, size=(n, L), dtype=np.uint64)
        hi = np.uint64(((1 << w) - 1) ^ ((1 << (w // 2)) - 1))
        flip = g.random(size=(n, L)) < 0.01
        x = np.where(flip, base, (base & ~hi) | (np.uint64(0x5A5A5A5A) & hi)).astype(dt)
        mask, bitval = o.build_meta(x, 0.9)
        slots, bitmask, row_bits = o.compress(x, B, mask, bitval)
        exp_bits = row_bits_formula(x, B, mask, bitval)
        assert np.array_equal(row_bits.astype(np.int64), exp_bits), (w, B, L)
        raw = L * w // 8
        exp_flag = 4 * ((exp_bits + 31) // 32) < raw
        got_flag = (bitmask[np.arange(n) // 32] >> (np.arange(n) % 32).astype(np.uint32)) & 1
        assert np.array_equal(got_flag.astype(bool), exp_flag), (w, B, L)
        idx = g.integers(0, n, size=100)
        out, rc = o.decompress_gather(slots, n, L, dt, B, bitmask, mask, bitval, idx)
        assert rc == 0 and np.array_equal(out, x[idx]), (w, B, L)


def check_positions_hand_example(o):
    """Per-position metadata on the hand-worked 8-bit rows (golden file)."""
    d = load_hand_example("positions_example_u8.txt", np.uint8)
    pm, pb = o.build_meta_positions(d["rows"], d["T"])
    assert pm.tolist() == d["pmask"] and pb.tolist() == d["pbitval"], (pm, pb)
    assert o.build_meta(d["rows"], d["T"]) == (0, 0)  # one shared mask finds nothing
    slots, bitmask, row_bits = o.compress_positions(d["rows"], d["block"], pm, pb)
    assert list(row_bits) == d["row_bits"]
    assert int(bitmask[0]) == d["bitmask"]
    for r, words in enumerate(d["streams"]):
        assert slots[r, :4].view("<u4").tolist() == words, (r, slots[r, :4].view("<u4"))
    typed = np.zeros_like(slots)
    for r, words in enumerate(d["streams"]):
        typed[r, :4] = np.array(words, dtype="<u4").view(np.uint8)
    idx = np.array([3, 0, 2, 1, 1])
    out, rc = o.decompress_gather_positions(typed, 4, 8, np.uint8, d["block"], bitmask,
                                            np.array(d["pmask"]), np.array(d["pbitval"]), idx)
    assert rc == 0 and np.array_equal(out, d["rows"][idx])


def check_positions_meta_and_sizes(o):
    """Per-position metadata equals the brute-force rule column by column; row sizes
    follow the size formula with per-element field widths; equal masks at every
    position reproduce the shared-mask stream byte for byte; round trips."""
    g = np.random.default_rng(2024)
    for dt, w, B, L in ((np.uint32, 32, 32, 64), (np.uint16, 16, 8, 40), (np.uint8, 8, 4, 22)):
        n = 60
        colconst = g.integers(0, 1 << w, size=L, dtype=np.uint64)
        colhi = np.array([((1 << w) - 1) ^ ((1 << int(k)) - 1) for k in
                          g.integers(1, w, size=L)], dtype=np.uint64)
        base = g.integers(0, 1 << w, size=(n, L), dtype=np.uint64)
        flip = g.random(size=(n, L)) < 0.02
        x = np.where(flip, base, (base & ~colhi) | (colconst & colhi)).astype(dt)
        for T in (0.9, 1.0):
            pm, pb = o.build_meta_positions(x, T)
            for e in range(L):
                assert (int(pm[e]), int(pb[e])) == brute_meta(x[:, e], T), (w, e)
            slots, bitmask, row_bits = o.compress_positions(x, B, pm, pb)
            m = w - np.array([bin(int(v)).count("1") for v in pm])
            ok = (x.astype(np.uint64) & pm.astype(np.uint64)) == pb.astype(np.uint64)
            bits = np.zeros(n, dtype=np.int64)
            for b0 in range(0, L, B):
                sl = slice(b0, min(b0 + B, L))
                match = ok[:, sl].all(axis=1)
                bits += 1 + np.where(match, m[sl].sum(), (sl.stop - sl.start) * w)
            assert np.array_equal(row_bits.astype(np.int64), bits), (w, T)
            idx = g.integers(0, n, size=80)
            out, rc = o.decompress_gather_positions(slots, n, L, dt, B, bitmask, pm, pb, idx)
            assert rc == 0 and np.array_equal(out, x[idx])
        # one mask repeated at every position = the shared-mask code
        mask, bitval = o.build_meta(x, 0.9)
        s1, b1, r1 = o.compress(x, B, mask, bitval)
        s2, b2, r2 = o.compress_positions(x, B, np.full(L, mask, np.uint32),
                                          np.full(L, bitval, np.uint32))
        assert np.array_equal(s1, s2) and np.array_equal(b1, b2) and np.array_equal(r1, r2)


def check_slot_bytes(o):
    """A slot is the raw row rounded up to 16 bytes."""
    for L, w, want in ((3, 32, 16), (4, 32, 16), (5, 32, 32), (8, 16, 16), (9, 16, 32),
                       (24, 8, 32), (16, 8, 16), (128, 32, 512), (11008, 16, 22016)):
        assert o.slot_bytes(L, w) == want, (L, w)


def check_code_cut_to_width(o):
    """The code of w-bit elements uses the low w bits of mask and bitval only: bits
    above w change nothing."""
    g = np.random.default_rng(31)
    x = g.integers(0, 1 << 16, size=(20, 64), dtype=np.uint64).astype(np.uint16)
    x[:10] = (x[:10] & np.uint16(0x00FF)) | np.uint16(0x3C00)
    a = o.compress(x, 32, 0xFF00, 0x3C00)
    b = o.compress(x, 32, 0xABCDFF00, 0x12343C00)
    assert all(np.array_equal(p, q) for p, q in zip(a, b))
    assert int(a[1][0]) != 0  # some rows compressed: the code is used


def check_decode_rejects_uncompressible_stream(o):
    """A slot flagged compressed whose participation bits describe a stream of at
    least the raw row's size is corrupt (such a row is always stored raw); one word
    less decodes. FP32, 32 elements, B = 16, mask of two bits (m = 30): header bits
    (raw, match) give 2 + 16*32 + 16*30 = 994 bits = 32 words = the 128 raw bytes;
    (match, match) give 2 + 2*16*30 = 962 bits = 31 words."""
    mask, bitval = 0xC0000000, 0x40000000
    for header, want in ((0b10, -6), (0b11, 0)):
        slots = np.zeros((1, 128), dtype=np.uint8)
        slots[0, 0] = header
        bm = np.array([1], dtype=np.uint32)
        out, rc = o.decompress_gather(slots, 1, 32, np.uint32, 16, bm, mask, bitval,
                                      np.array([0]))
        assert rc == want, (header, rc)


def check_bad_index_semantics(o):
    """A gather rebuilds every valid index even after a bad one; each bad index
    (negative or past the table) leaves its output row untouched and makes the call
    report a bad index. The same holds for the packed store's gather."""
    rows = np.arange(8 * 32, dtype=np.uint32).reshape(8, 32) | np.uint32(0x3F000000)
    mask, bitval = o.build_meta(rows, 0.9)
    slots, bitmask, row_bits = o.compress(rows, 32, mask, bitval)
    idx = np.array([3, -1, 0, 8, 7, 1 << 40, 3], dtype=np.int64)
    good = [0, 2, 4, 6]
    sentinel = np.full((idx.size, 32), 0xDEADBEEF, dtype=np.uint32)
    out, rc = o.decompress_gather(slots, 8, 32, np.uint32, 32, bitmask, mask, bitval, idx,
                                  out=sentinel.copy())
    assert rc == -5, rc
    assert np.array_equal(out[good], rows[idx[good]])
    assert np.all(out[[1, 3, 5]] == 0xDEADBEEF)
    off, packed, pbm, _ = o.pack(slots, 32, np.uint32, bitmask, row_bits)
    out, rc = o.decompress_gather_packed(packed, off, 32, np.uint32, 32, pbm, mask, bitval, idx,
                                         out=sentinel.copy())
    assert rc == -5, rc
    assert np.array_equal(out[good], rows[idx[good]])
    assert np.all(out[[1, 3, 5]] == 0xDEADBEEF)


def check_stream_padding_is_zero(o):
    """The stored bytes of a compressed row are its stream and zero bits up to the
    end of the last 32-bit word, whatever the slot held before: compressing into a
    buffer full of ones gives the same used prefix as into a zeroed one."""
    g = np.random.default_rng(12)
    x = (g.integers(0, 1 << 20, size=(40, 96), dtype=np.uint64).astype(np.uint32)
         | np.uint32(0x3F800000))
    mask, bitval = o.build_meta(x, 0.9)
    clean, bm, rb = o.compress(x, 32, mask, bitval)
    dirty = np.full_like(clean, 0xFF)
    bm2 = np.zeros_like(bm)
    rb2 = np.zeros_like(rb)
    rc = o.lib.ibpo_compress(x.ctypes.data, 40, 96, 32, 32, int(mask), int(bitval),
                             dirty.ctypes.data, clean.shape[1], bm2.ctypes.data, rb2.ctypes.data)
    assert rc == 0 and np.array_equal(bm, bm2) and np.array_equal(rb, rb2)
    comp = [(bm[r // 32] >> (r % 32)) & 1 for r in range(40)]
    assert any(comp)
    for r in range(40):
        used = 4 * ((int(rb[r]) + 31) // 32) if comp[r] else 96 * 4
        assert np.array_equal(dirty[r, :used], clean[r, :used]), r


def check_size_formula(o):
    g = np.random.default_rng(777)
    cases = [(np.uint32, 32, 32, 128), (np.uint32, 32, 64, 256), (np.uint16, 16, 64, 256),
             (np.uint16, 16, 32, 96), (np.uint32, 32, 4, 12), (np.uint16, 16, 1, 5)]
    for dt, w, B, L in cases:
        n = 64
        base = g.integers(0, 1 << w, size=(n, L), dtype=np.uint64)
        # high bits mostly constant so that most blocks match
        hi = np.uint64(((1 << w) - 1) ^ ((1 << (w // 2)) - 1))
        flip = g.random(size=(n, L)) < 0.01
        x = np.where(flip, base, (base & ~hi) | (np.uint64(0x5A5A5A5A) & hi)).astype(dt)
        mask, bitval = o.build_meta(x, 0.9)
        slots, bitmask, row_bits = o.compress(x, B, mask, bitval)
        m = w - bin(mask).count("1")
        match = block_matches(x, B, mask, bitval)
        exp_bits = (1 + np.where(match, B * m, B * w)).sum(axis=1)
        assert np.array_equal(row_bits.astype(np.int64), exp_bits)
        raw = L * w // 8
        exp_flag = 4 * ((exp_bits + 31) // 32) < raw
        got_flag = ((bitmask[np.arange(n) // 32] >> (np.arange(n) % 32).astype(np.uint32)) & 1)
        assert np.array_equal(got_flag.astype(bool), exp_flag)
    # equality case of the store rule: FP32, B = L = 32, only the sign bit
    # invariant -> 1 + 32*31 = 993 bits = 32 words = 128 B = raw -> stored raw
    x = g.integers(0, 1 << 31, size=(8, 32), dtype=np.uint64).astype(np.uint32)
    x[:, 0] = 0x7FFFFFFF
    x[:, 1] = 0x00000000
    mask, bitval = o.build_meta(x, 1.0)
    assert mask == 0x80000000 and bitval == 0
    slots, bitmask, row_bits = o.compress(x, 32, mask, bitval)
    assert np.all(row_bits == 993)
    assert int(bitmask[0]) == 0
    assert np.array_equal(slots[:, :128].view("<u4"), x)


def expected_slot_bits(row: np.ndarray, B: int, mask: int, bitval: int) -> str:
    """The row's stream as a string of '0'/'1' characters, stream bit i at index i."""
    w = 8 * row.dtype.itemsize
    L = row.size
    kept = [j for j in range(w) if not (mask >> j) & 1]
    blocks = [row[b * B:(b + 1) * B] for b in range(L // B)]
    parts = []
    flags = [all((int(x) & mask) == bitval for x in blk) for blk in blocks]
    parts.append("".join("1" if f else "0" for f in flags))
    for f, blk in zip(flags, blocks):
        for x in blk:
            x = int(x)
            if f:
                parts.append("".join(str((x >> j) & 1) for j in kept))
            else:
                parts.append("".join(str((x >> j) & 1) for j in range(w)))
    return "".join(parts)


def words_from_bitstring(s: str) -> list[int]:
    s = s + "0" * (-len(s) % 32)
    return [int(s[i:i + 32][::-1], 2) for i in range(0, len(s), 32)]


def check_stream_layout(o):
    g = np.random.default_rng(4242)
    for dt, w, B, L in ((np.uint16, 16, 4, 16), (np.uint32, 32, 8, 24), (np.uint16, 16, 2, 6),
                        (np.uint32, 32, 32, 64)):
        n = 12
        base = g.integers(0, 1 << w, size=(n, L), dtype=np.uint64)
        keep_hi = np.uint64(((1 << w) - 1) ^ ((1 << (w // 2 - 3)) - 1))
        flip = g.random(size=(n, L)) < 0.05
        x = np.where(flip, base, (base & ~keep_hi) | (np.uint64(0x3C3C3C3C) & keep_hi)).astype(dt)
        mask, bitval = o.build_meta(x, 0.8)
        slots, bitmask, row_bits = o.compress(x, B, mask, bitval)
        raw = L * w // 8
        for r in range(n):
            s = expected_slot_bits(x[r], B, mask, bitval)
            assert len(s) == int(row_bits[r])
            compressed = (int(bitmask[r // 32]) >> (r % 32)) & 1
            if compressed:
                words = words_from_bitstring(s)
                assert slots[r, : 4 * len(words)].view("<u4").tolist() == words
            else:
                assert bytes(slots[r, :raw]) == x[r].tobytes()


def special_words(w: int) -> list[int]:
    if w == 8:  # FP8 E4M3 / E5M2 patterns: +-0, denormals, NaN/Inf encodings, all-ones
        return [0x00, 0x80, 0x01, 0x07, 0x81, 0x7F, 0xFF, 0x7C, 0xFC, 0x7E, 0x38, 0xB8, 0x08,
                0x3C]
    if w == 32:
        return [0x00000000, 0x80000000, 0x00000001, 0x007FFFFF, 0x80000001, 0x7F800000,
                0xFF800000, 0x7FC00000, 0x7FC12345, 0x7F800001, 0xFFFFFFFF, 0x3F800000,
                0xBF800000, 0x00800000]
    return [0x0000, 0x8000, 0x0001, 0x03FF, 0x8001, 0x7C00, 0xFC00, 0x7E00, 0x7E5A, 0x7C01,
            0xFFFF, 0x3C00, 0xBC00, 0x7F80, 0xFF80, 0x7FC1, 0x0400]


def check_round_trip_specials(o):
    g = np.random.default_rng(99)
    for dt, w in ((np.uint32, 32), (np.uint16, 16), (np.uint8, 8)):
        sp = np.array(special_words(w), dtype=dt)
        for B in (1, 2, 4, 8, 32):
            L = B * 4
            n = 40
            x = sp[g.integers(0, sp.size, size=(n, L))]
            # rows that are mostly one special word, so that blocks also match
            x[: n // 2] = np.where(g.random(size=(n // 2, L)) < 0.9, sp[g.integers(0, sp.size)],
                                   x[: n // 2])
            for T in (0.0, 0.6, 0.9, 1.0):
                mask, bitval = o.build_meta(x, T)
                for mk, bv in ((mask, bitval), (0, 0), (wmask(w), int(x[0, 0])),
                               (0x7F80 if w == 16 else 0x7F800000, 0)):
                    slots, bitmask, _ = o.compress(x, B, mk, bv & mk)
                    idx = g.integers(0, n, size=64)
                    out, rc = o.decompress_gather(slots, n, L, dt, B, bitmask, mk, bv & mk, idx)
                    assert rc == 0
                    assert np.array_equal(out, x[idx]), (w, B, T, hex(mk))


def load_select_examples():
    out, cur = {}, None
    with open(os.path.join(GOLDEN, "select_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "example":
                cur = out.setdefault(vals[0], {})
            elif key == "T":
                cur["T"] = float(vals[0])
            elif key == "block":
                cur["block"] = int(vals[0])
            elif key == "candidates":
                cur["candidates"] = [(int(v.split(":")[0], 16), int(v.split(":")[1]))
                                     for v in vals]
            elif key == "choice":
                cur["choice"] = (int(vals[0], 16), int(vals[1], 16))
    return out


def fp32_bit26_rows() -> np.ndarray:
    """The formula of the fp32_bit26 example: one bit-26 exception per row."""
    r = np.arange(8, dtype=np.uint32)[:, None]
    e = np.arange(32, dtype=np.uint32)[None, :]
    return (np.uint32(0x38000000) | np.where(e == r, np.uint32(1 << 26), np.uint32(0))
            | (e << np.uint32(3)) | (r & np.uint32(7))).astype(np.uint32)


def check_select_examples(o):
    ex = load_select_examples()
    rows = {"fp16_hand": load_hand_example()["rows"], "fp32_bit26": fp32_bit26_rows()}
    for name, d in ex.items():
        mask, bitval, cands = o.select_meta(rows[name], d["T"], d["block"])
        assert cands == d["candidates"], (name, [(hex(m), b) for m, b in cands])
        assert (mask, bitval) == d["choice"], (name, hex(mask), hex(bitval))


def stored_total(rows: np.ndarray, B: int, mask: int, bitval: int) -> int:
    """Bytes the rows take under (mask, bitval), from the size formula alone."""
    n, L = rows.shape
    w = 8 * rows.dtype.itemsize
    m = w - bin(mask).count("1")
    bits = (1 + np.where(block_matches(rows, B, mask, bitval), B * m, B * w)).sum(axis=1)
    words = (bits + 31) // 32
    raw = L * w // 8
    return int(np.where(4 * words < raw, 4 * words, raw).sum())


def threshold_family(rows: np.ndarray, T: float):
    """Every distinct mask of the threshold rule at thresholds >= T (counts are
    integers, so thresholds halfway between them reach every mask), plus the empty
    mask; each with bitval = the majority values of its positions."""
    N = rows.size
    masks = {}
    for T2 in [T] + [(c - 0.5) / N for c in range(1, N + 1) if (c - 0.5) / N >= T]:
        mk, bv = brute_meta(rows, T2)
        masks[mk] = bv
    masks.setdefault(0, 0)
    return masks


def check_select_threshold_sweep(o):
    g = np.random.default_rng(4242)
    cases = []
    for trial in range(24):
        dt, w = ((np.uint16, 16), (np.uint32, 32))[trial % 2]
        B = (1, 2, 4, 8)[trial % 4]
        n, L = int(g.integers(1, 9)), B * int(g.integers(1, 5))
        base = g.integers(0, 1 << w, size=(n, L), dtype=np.uint64)
        hi = np.uint64(((1 << w) - 1) ^ ((1 << (w // 4)) - 1))
        flip = g.random(size=(n, L)) < (0.0, 0.03, 0.1, 0.5)[trial % 4 if trial < 20 else 3]
        const = np.uint64(int(g.integers(0, 1 << w)))
        x = np.where(flip, base, (base & ~hi) | (const & hi)).astype(dt)
        # one exception per row in a high position that the threshold rule keeps
        if trial % 3 == 0:
            x[:, 0] ^= dt(1 << (w - 3))
        cases.append((x, float((0.5, 0.75, 0.9)[trial % 3]), B))
    for x, T, B in cases:
        fam = threshold_family(x, T)
        scored = sorted(((stored_total(x, B, mk, bv), -bin(mk).count("1"), mk, bv)
                         for mk, bv in fam.items()))
        best_bytes, _, best_mask, best_bitval = scored[0]
        mask, bitval, cands = o.select_meta(x, T, B)
        assert (mask, bitval) == (best_mask, best_bitval), (hex(mask), hex(best_mask), T, B)
        assert sorted(m for m, _ in cands) == sorted(fam), ([hex(m) for m, _ in cands],
                                                            [hex(m) for m in fam])
        for mk, b in cands:
            assert b == stored_total(x, B, mk, fam[mk])
        assert dict(cands)[mask] == best_bytes


def check_pack_hand_example(o):
    """Rows 1, 0, 1 of the hand-worked example packed end to end: each entry is the
    row's stream words (typed in from the golden file) padded to 16 bytes."""
    d = load_hand_example()
    n, L = d["rows"].shape
    slots = np.zeros((n, 16), dtype=np.uint8)
    for r, words in enumerate(d["streams"]):
        slots[r, : 4 * len(words)] = np.array(words, dtype="<u4").view(np.uint8)
    bitmask = np.array([d["bitmask"]], dtype=np.uint32)
    row_bits = np.array(d["row_bits"], dtype=np.uint32)
    sel = np.array([1, 0, 1], dtype=np.int64)
    offsets, packed, pbm, prb = o.pack(slots, L, np.uint16, bitmask, row_bits, sel)
    # row0: 50 bits -> 8 B -> 16; row1: 90 bits -> 12 B -> 16
    assert offsets.tolist() == [0, 16, 32, 48]
    for i, r in enumerate(sel):
        words = d["streams"][r]
        assert packed[16 * i: 16 * i + 4 * len(words)].view("<u4").tolist() == words
    assert int(pbm[0]) == 0b111
    assert prb.tolist() == [90, 50, 90]
    out, rc = o.decompress_gather_packed(packed, offsets, L, np.uint16, d["block"], pbm,
                                         d["mask"], d["bitval"], np.array([2, 1, 0, 1]))
    assert rc == 0
    assert np.array_equal(out, d["rows"][[1, 0, 1, 0]])


def check_pack_round_trip(o):
    g = np.random.default_rng(99)
    for dt, w, B, L in ((np.uint32, 32, 32, 128), (np.uint16, 16, 64, 256), (np.uint32, 32, 4, 36)):
        n = 120
        base = g.integers(0, 1 << w, size=(n, L), dtype=np.uint64)
        hi = np.uint64(((1 << w) - 1) ^ ((1 << (w // 2)) - 1))
        flip = g.random(size=(n, L)) < 0.004
        x = np.where(flip, base, (base & ~hi) | (np.uint64(0x3C1E3C1E) & hi)).astype(dt)
        x[::7] = base[::7].astype(dt)  # some rows stored raw
        mask, bitval = o.build_meta(x, 0.9)
        slots, bitmask, row_bits = o.compress(x, B, mask, bitval)
        sel = g.integers(0, n, size=200)
        offsets, packed, pbm, prb = o.pack(slots, L, dt, bitmask, row_bits, sel)
        # entry sizes from the size formula alone
        m = w - bin(mask).count("1")
        bits = (1 + np.where(block_matches(x, B, mask, bitval), B * m, B * w)).sum(axis=1)
        words = (bits + 31) // 32
        raw = L * w // 8
        used = np.where(4 * words < raw, 4 * words, raw)
        sizes = (used[sel] + 15) // 16 * 16
        assert np.array_equal(np.diff(offsets), sizes)
        assert offsets[0] == 0 and packed.size == sizes.sum()
        idx = g.integers(0, sel.size, size=300)
        out, rc = o.decompress_gather_packed(packed, offsets, L, dt, B, pbm, mask, bitval, idx)
        assert rc == 0
        assert np.array_equal(out, x[sel[idx]])
        # an entry cut short is corrupt, and its output row is left alone
        i = int(np.nonzero(np.diff(offsets) >= 32)[0][0])
        bad = offsets.copy()
        bad[i + 1] = bad[i] + 16 * ((int(used[sel[i]]) - 1) // 16)  # one 16-byte piece short
        sentinel = np.full((1, L), 7, dtype=dt)
        out, rc = o.decompress_gather_packed(packed, bad, L, dt, B, pbm, mask, bitval,
                                             np.array([i]), out=sentinel.copy())
        assert rc == -6 and np.array_equal(out, sentinel)


def check_block_positions_hand_example(o):
    """Block-position metadata on the hand-worked 8-bit rows with a shorter last
    block (golden file), and compression with the tiled tables."""
    d = load_hand_example("block_positions_example_u8.txt", np.uint8)
    pm, pb = o.build_meta_block_positions(d["rows"], d["T"], d["block"])
    assert pm.tolist() == d["pmask"] and pb.tolist() == d["pbitval"], (pm, pb)
    slots, bitmask, row_bits = o.compress_positions(d["rows"], d["block"], pm, pb)
    assert list(row_bits) == d["row_bits"]
    assert int(bitmask[0]) == d["bitmask"]
    for r, words in enumerate(d["streams"]):
        assert slots[r, :4].view("<u4").tolist() == words, (r, slots[r, :4].view("<u4"))
    out, rc = o.decompress_gather_positions(slots, 2, 6, np.uint8, d["block"], bitmask, pm, pb,
                                            np.array([1, 0, 1]))
    assert rc == 0 and np.array_equal(out, d["rows"][[1, 0, 1]])


def check_block_positions_reductions(o):
    """Block-position metadata: position q is the brute-force rule over the
    elements q, q + B, q + 2B, ... of every row, and every element takes its
    position's pair; with B = 1 it is the shared mask, with B >= L the per-element
    metadata. Rows with and without a shorter last block."""
    g = np.random.default_rng(77)
    for dt, w, B, L in ((np.uint32, 32, 8, 40), (np.uint16, 16, 16, 56), (np.uint8, 8, 4, 22),
                        (np.uint8, 8, 32, 32)):
        n = 50
        colconst = g.integers(0, 1 << w, size=B, dtype=np.uint64)
        colhi = np.array([((1 << w) - 1) ^ ((1 << int(k)) - 1) for k in
                          g.integers(1, w, size=B)], dtype=np.uint64)
        base = g.integers(0, 1 << w, size=(n, L), dtype=np.uint64)
        q_of = np.arange(L) % B
        flip = g.random(size=(n, L)) < 0.05
        x = np.where(flip, base, (base & ~colhi[q_of]) | (colconst[q_of] & colhi[q_of]))
        x = x.astype(dt)
        for T in (0.8, 0.95, 1.0):
            pm, pb = o.build_meta_block_positions(x, T, B)
            for q in range(min(B, L)):
                want = brute_meta(x[:, q::B], T)
                assert all((int(pm[e]), int(pb[e])) == want for e in range(q, L, B)), (w, q)
            assert (o.build_meta_block_positions(x, T, 1)[0] == o.build_meta(x, T)[0]).all()
            assert (o.build_meta_block_positions(x, T, 1)[1] == o.build_meta(x, T)[1]).all()
            for BB in (L, L + 5):
                a = o.build_meta_block_positions(x, T, BB)
                b = o.build_meta_positions(x, T)
                assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


ALL_CHECKS = [check_hand_example, check_hand_decode, check_meta_exhaustive,
              check_meta_closed_forms, check_size_formula, check_stream_layout,
              check_round_trip_specials, check_select_examples,
              check_select_threshold_sweep, check_pack_hand_example, check_pack_round_trip,
              check_hand_example_u8_tail, check_tail_blocks_and_bytes,
              check_positions_hand_example, check_positions_meta_and_sizes,
              check_block_positions_hand_example, check_block_positions_reductions,
              check_slot_bytes, check_code_cut_to_width,
              check_decode_rejects_uncompressible_stream, check_bad_index_semantics,
              check_stream_padding_is_zero]
