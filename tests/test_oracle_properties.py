"""Properties of the oracle on random inputs (no GPU; needs hypothesis, skipped
where it is not installed).

For random element widths, block sizes (any B >= 1, not only the GPU's), row
lengths (shorter last blocks included), masks, bitvals and thresholds:
  * decompress-gather rebuilds every row bit for bit;
  * each row's bit count is the size formula, and a row is stored compressed
    exactly when its stream needs fewer bytes than the raw row;
  * the metadata is the brute-force rule;
  * the per-position and block-position codes round-trip, and the packed store
    gathers what the slotted store gathers.
"""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402
import pins  # noqa: E402

DT = {8: np.uint8, 16: np.uint16, 32: np.uint32}


@st.composite
def tables(draw):
    w = draw(st.sampled_from([8, 16, 32]))
    n = draw(st.integers(1, 12))
    L = draw(st.integers(1, 70))
    B = draw(st.integers(1, 40))
    seed = draw(st.integers(0, 2 ** 32 - 1))
    g = np.random.default_rng(seed)
    hi_bits = draw(st.integers(0, w))
    flip = draw(st.sampled_from([0.0, 0.01, 0.1, 0.5]))
    top = ((1 << w) - 1) ^ ((1 << (w - hi_bits)) - 1) if hi_bits else 0
    const = int(g.integers(0, 1 << w))
    base = g.integers(0, 1 << w, size=(n, L), dtype=np.uint64)
    keep = g.random(size=(n, L)) >= flip
    rows = np.where(keep, (base & ~np.uint64(top)) | np.uint64(const & top), base)
    return rows.astype(DT[w]), w, B


@settings(max_examples=300, deadline=None)
@given(tables(), st.sampled_from([0.5, 0.7, 0.9, 1.0]))
def test_threshold_code_round_trip_and_sizes(t, T):
    rows, w, B = t
    o = oracle.default()
    n, L = rows.shape
    mask, bitval = o.build_meta(rows, T)
    assert (mask, bitval) == pins.brute_meta(rows, T)
    slots, bitmask, row_bits = o.compress(rows, B, mask, bitval)
    assert np.array_equal(row_bits.astype(np.int64), pins.row_bits_formula(rows, B, mask, bitval))
    comp = (bitmask[np.arange(n) // 32] >> (np.arange(n) % 32).astype(np.uint32)) & 1
    raw = L * w // 8
    assert np.array_equal(comp == 1, 4 * ((row_bits.astype(np.int64) + 31) // 32) < raw)
    idx = np.arange(n)[::-1].copy()
    out, rc = o.decompress_gather(slots, n, L, rows.dtype, B, bitmask, mask, bitval, idx)
    assert rc == 0 and np.array_equal(out, rows[idx])
    off, packed, pbm, _ = o.pack(slots, L, rows.dtype, bitmask, row_bits)
    out2, rc = o.decompress_gather_packed(packed, off, L, rows.dtype, B, pbm, mask, bitval, idx)
    assert rc == 0 and np.array_equal(out2, rows[idx])


@settings(max_examples=300, deadline=None)
@given(tables(), st.integers(0, 2 ** 32 - 1))
def test_any_code_round_trips(t, code_seed):
    """Any mask/bitval pair is a valid code, also one the rows rarely match."""
    rows, w, B = t
    o = oracle.default()
    n, L = rows.shape
    g = np.random.default_rng(code_seed)
    mask = int(g.integers(0, 1 << w))
    bitval = int(g.integers(0, 1 << w)) & mask
    slots, bitmask, row_bits = o.compress(rows, B, mask, bitval)
    assert np.array_equal(row_bits.astype(np.int64), pins.row_bits_formula(rows, B, mask, bitval))
    out, rc = o.decompress_gather(slots, n, L, rows.dtype, B, bitmask, mask, bitval,
                                  np.arange(n))
    assert rc == 0 and np.array_equal(out, rows)


@settings(max_examples=150, deadline=None)
@given(tables(), st.sampled_from([0.6, 0.9, 1.0]))
def test_position_codes_round_trip(t, T):
    rows, w, B = t
    o = oracle.default()
    n, L = rows.shape
    for pm, pb in (o.build_meta_positions(rows, T), o.build_meta_block_positions(rows, T, B)):
        slots, bitmask, row_bits = o.compress_positions(rows, B, pm, pb)
        out, rc = o.decompress_gather_positions(slots, n, L, rows.dtype, B, bitmask, pm, pb,
                                                np.arange(n))
        assert rc == 0 and np.array_equal(out, rows)
    # block positions are periodic in B and follow the rule over their own sample
    pm, pb = o.build_meta_block_positions(rows, T, B)
    for q in range(min(B, L)):
        want = pins.brute_meta(rows[:, q::B], T)
        assert all((int(pm[e]), int(pb[e])) == want for e in range(q, L, B))
