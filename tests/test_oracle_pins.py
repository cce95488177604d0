"""The oracle against what the method and mathematics fix (no GPU needed)."""
import numpy as np
import pytest

import ibp_inputs as gen
import oracle
import pins


@pytest.fixture(scope="module")
def o():
    return oracle.default()


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(o, check):
    check(o)


def test_brute_meta_on_workload_prefixes(o):
    cases = [(gen.tiny_fp32(512), 0.9), (gen.gnn_dense(300), 0.9), (gen.gnn_sparse(40), 0.9),
             (gen.dlrm_table(3, 300), 0.95), (gen.llm_weight(0, "q", 16), 0.9),
             (gen.llm_kv(1, 1, n_rows=8), 0.9)]
    for x, T in cases:
        words = x.view(np.uint32) if x.dtype == np.float32 else x
        assert o.build_meta(words, T) == pins.brute_meta(words, T)


@pytest.mark.parametrize("name,B,T", [("tiny", 32, 0.9), ("dense", 32, 0.9), ("sparse", 32, 0.9),
                                      ("dlrm", 32, 0.95), ("w_down", 64, 0.9), ("kv", 64, 0.9)])
def test_round_trip_workload_prefixes(o, name, B, T):
    x = {"tiny": lambda: gen.tiny_fp32(1024), "dense": lambda: gen.gnn_dense(1000),
         "sparse": lambda: gen.gnn_sparse(200), "dlrm": lambda: gen.dlrm_table(0, 1000),
         "w_down": lambda: gen.llm_weight(2, "down", 24),
         "kv": lambda: gen.llm_kv(0, 0, n_rows=64)}[name]()
    words = x.view(np.uint32) if x.dtype == np.float32 else x
    mask, bitval = o.build_meta(words, T)
    slots, bitmask, row_bits = o.compress(words, B, mask, bitval)
    n, L = words.shape
    g = np.random.default_rng(5)
    idx = np.concatenate([g.integers(0, n, size=300), [0, n - 1, n - 1, 0]]).astype(np.int64)
    out, rc = o.decompress_gather(slots, n, L, words.dtype, B, bitmask, mask, bitval, idx)
    assert rc == 0
    assert np.array_equal(out, words[idx])
    match = pins.block_matches(words, B, mask, bitval)
    m = 8 * words.dtype.itemsize - bin(mask).count("1")
    exp = (1 + np.where(match, B * m, B * 8 * words.dtype.itemsize)).sum(axis=1)
    assert np.array_equal(row_bits.astype(np.int64), exp)


def test_error_paths(o):
    x = gen.tiny_fp32(64).view(np.uint32)
    mask, bitval = o.build_meta(x, 0.9)
    slots, bitmask, _ = o.compress(x, 32, mask, bitval)
    n, L = x.shape
    sentinel = np.full((3, L), 0xDEADBEEF, dtype=np.uint32)
    out, rc = o.decompress_gather(slots, n, L, np.uint32, 32, bitmask, mask, bitval,
                                  np.array([1, n, -1], dtype=np.int64), out=sentinel.copy())
    assert rc == oracle.BAD_INDEX
    assert np.array_equal(out[0], x[1])
    assert np.all(out[1:] == 0xDEADBEEF)
    # corrupt a compressed row: participation bits all 0 describe a raw-sized stream
    r = next(r for r in range(n) if (bitmask[r // 32] >> (r % 32)) & 1)
    bad = slots.copy()
    bad[r, 0] &= 0xF0
    out, rc = o.decompress_gather(bad, n, L, np.uint32, 32, bitmask, mask, bitval,
                                  np.array([r], dtype=np.int64), out=sentinel[:1].copy())
    assert rc == oracle.CORRUPT
    assert np.all(out == 0xDEADBEEF)
    # empty gather is a no-op
    out, rc = o.decompress_gather(slots, n, L, np.uint32, 32, bitmask, mask, bitval,
                                  np.zeros(0, dtype=np.int64))
    assert rc == 0 and out.shape == (0, L)


# Mistakes planted in a copy of the oracle source; each must break at least one pin.
PLANTED = [
    ("threshold > instead of >=", "(double)cv >= T * (double)n_elems",
     "(double)cv > T * (double)n_elems"),
    ("tie picks 1", "int v = c1 > c0 ? 1 : 0;", "int v = c1 >= c0 ? 1 : 0;"),
    ("participation bit dropped from size",
     "bits += 1 + block_payload_bits(c, b, row_elems, block_elems, w_bits, match);",
     "bits += block_payload_bits(c, b, row_elems, block_elems, w_bits, match);"),
    ("tail block sized as a full block",
     "const int64_t len = block_len(b, row_elems, block_elems);",
     "const int64_t len = block_elems;"),
    ("kept bits taken from the mask", "    if (!bit_of(mask, j)) {\n      field",
     "    if (bit_of(mask, j)) {\n      field"),
    ("MSB-first bit order", "  int in_word = (int)(pos % 32);\n  int64_t byte = word * 4 + in_word / 8;\n  int in_byte = in_word % 8;\n  if (bit)",
     "  int in_word = 31 - (int)(pos % 32);\n  int64_t byte = word * 4 + in_word / 8;\n  int in_byte = in_word % 8;\n  if (bit)"),
    ("store rule <= instead of <", "int compressed = 4 * stored_words < raw_bytes;",
     "int compressed = 4 * stored_words <= raw_bytes;"),
    ("payload read starts one bit late", "int64_t pos = nb; /* first payload bit */",
     "int64_t pos = nb + 1; /* first payload bit */"),
    ("bitval not reinserted", "x |= (uint32_t)bit_of(bitval, j) << j;", "x |= 0;"),
    ("bitval stores the minority value", "bitval |= (uint32_t)v << j;",
     "bitval |= (uint32_t)(1 - v) << j;"),
    ("selection ties go to the smaller mask", "if (total[k] < total[best]) best = k;",
     "if (total[k] <= total[best]) best = k;"),
    ("selection drops the most-held positions first",
     "if (bit_of(cur, j) && (fewest < 0 || held[j] < fewest)) fewest = held[j];",
     "if (bit_of(cur, j) && (fewest < 0 || held[j] > fewest)) fewest = held[j];"),
    ("selection drops tied positions one at a time",
     "if (bit_of(cur, j) && held[j] == fewest) cur &= ~(1u << j);",
     "if (bit_of(cur, j) && held[j] == fewest) { cur &= ~(1u << j); break; }"),
    ("packed entries rounded to 4 bytes", "int64_t len = (used + 15) / 16 * 16;",
     "int64_t len = (used + 3) / 4 * 4;"),
    ("packed entry length not checked",
     "if (4 * ((bits + 31) / 32) >= raw_bytes || 4 * ((bits + 31) / 32) > avail) return IBPO_CORRUPT;",
     "if (4 * ((bits + 31) / 32) >= raw_bytes) return IBPO_CORRUPT;"),
    ("positions use the first position's mask",
     "uint32_t mk = (shared ? pmask[0] : pmask[e]) & width_mask(w_bits);",
     "uint32_t mk = (shared ? pmask[0] : pmask[0]) & width_mask(w_bits);"),
    ("positions metadata samples position 0 only",
     "column[(size_t)(r * nbytes + k)] = base[(r * row_elems + e) * nbytes + k];",
     "column[(size_t)(r * nbytes + k)] = base[(r * row_elems) * nbytes + k];"),
    ("block positions sample only the first block",
     "      for (int64_t e = q; e < row_elems; e += block_elems)\n        for (int k = 0; k < nbytes; ++k) sample",
     "      for (int64_t e = q; e < row_elems && e < block_elems; e += block_elems)\n        for (int k = 0; k < nbytes; ++k) sample"),
    ("block positions tiled by block index",
     "    for (int64_t e = q; e < row_elems; e += block_elems) {\n      pmask_out[e] = mask;",
     "    for (int64_t e = q * block_elems; e < row_elems && e < (q + 1) * block_elems; ++e) {\n      pmask_out[e] = mask;"),
    ("block positions count a shorter last block as full",
     "    int rc = ibpo_build_meta(sample.data(), (int64_t)(sample.size() / nbytes), w_bits, T, &mask,",
     "    while ((int64_t)(sample.size() / nbytes) < n_rows * ((row_elems + block_elems - 1) / block_elems))\n      for (int k = 0; k < nbytes; ++k) sample.push_back(0);\n    int rc = ibpo_build_meta(sample.data(), (int64_t)(sample.size() / nbytes), w_bits, T, &mask,"),
    ("decoder accepts a stream of the raw size", "if (4 * ((bits + 31) / 32) >= raw_bytes ||",
     "if (4 * ((bits + 31) / 32) > raw_bytes ||"),
    ("code not cut to the element width",
     "uint32_t mk = (shared ? pmask[0] : pmask[e]) & width_mask(w_bits);",
     "uint32_t mk = (shared ? pmask[0] : pmask[e]);"),
    ("slot rounded to 8 bytes", "return (raw + 15) / 16 * 16;", "return (raw + 7) / 8 * 8;"),
    ("big-endian element load", "v |= (uint32_t)base[e * nbytes + k] << (8 * k);",
     "v |= (uint32_t)base[e * nbytes + k] << (8 * (nbytes - 1 - k));"),
    ("fields read MSB-first", "    v |= (uint32_t)get_bit(stream, *pos) << i;",
     "    v |= (uint32_t)get_bit(stream, *pos) << (nbits - 1 - i);"),
    ("block match tests the block's first position only",
     "    if ((load_elem(row, e, w_bits) & c.mask[e]) != c.bitval[e]) match = 0;",
     "    if ((load_elem(row, e, w_bits) & c.mask[b * block_elems]) != c.bitval[b * block_elems]) match = 0;"),
    ("gather stops at the first bad index",
     "      if (status == IBPO_OK) status = IBPO_BAD_INDEX;\n      continue;\n    }\n    int compressed = (int)((bitmask[r / 32] >> (r % 32)) & 1u);\n    int rc = decode_row(",
     "      if (status == IBPO_OK) status = IBPO_BAD_INDEX;\n      break;\n    }\n    int compressed = (int)((bitmask[r / 32] >> (r % 32)) & 1u);\n    int rc = decode_row("),
    ("gather reports a bad index as success",
     "    if (r < 0 || r >= n_rows) {\n      if (status == IBPO_OK) status = IBPO_BAD_INDEX;\n      continue;\n    }\n    int compressed = (int)((bitmask[r / 32] >> (r % 32)) & 1u);\n    int rc = decode_row(",
     "    if (r < 0 || r >= n_rows) {\n      continue;\n    }\n    int compressed = (int)((bitmask[r / 32] >> (r % 32)) & 1u);\n    int rc = decode_row("),
    ("compressed slot not cleared to the end of its last word",
     "    for (int64_t k = 0; k < 4 * stored_words; ++k) slot[k] = 0;",
     "    for (int64_t k = 0; k < 4 * stored_words - 1; ++k) slot[k] = 0;"),
    ("selection keeps the threshold bitval", "*bitval_out = bitval0 & cands[best];",
     "*bitval_out = bitval0;"),
]


@pytest.mark.parametrize("label,old,new", PLANTED, ids=[p[0] for p in PLANTED])
def test_planted_mistake_is_caught(tmp_path, label, old, new):
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation anchor not found once: {label}"
    bad = oracle.compile_variant(src.replace(old, new), str(tmp_path))
    failures = []
    for check in pins.ALL_CHECKS:
        try:
            check(bad)
        except AssertionError:
            failures.append(check.__name__)
    assert failures, f"planted mistake '{label}' passed every pin"
