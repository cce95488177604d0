/*
 * Plain single-threaded CPU oracle for Invariant Bit Packing (IBP).
 * TEST INFRASTRUCTURE ONLY (see ibp_oracle.h): nothing in the GPU codec uses it.
 *
 * Written for obviousness, not speed: every bit is moved by its own loop
 * iteration, elements are assembled byte by byte in little-endian order, and the
 * steps follow the order in which the IBP page ("Reducing the GPU Memory
 * Bottleneck with Lossless Compression for ML -- Extended", technical summary)
 * states them: preprocessing -> compression -> decompression.
 *
 * Readings of points the page leaves open (also listed in the design notes):
 *  R1 one w-bit mask/bitval pair applies to every element word;
 *  R2 all participation bits of a row come first, then the block payloads (the
 *     page prepends the bit per block and scans block sizes with a prefix scan;
 *     a header-first layout gives the same bit count and lets the scan start at once);
 *  R3 LSB-first bit order inside little-endian 32-bit words; a field holds the
 *     element's non-invariant bits in ascending position order;
 *  R4 bit j is invariant iff count(majority value) >= T*N in IEEE double;
 *  R5 majority value on a tie is 0;
 *  R6 with an empty mask every block "matches" and costs B*w bits anyway;
 *  R7 a row is kept compressed only when its stream needs fewer whole 32-bit
 *     words than the raw row has bytes / 4;
 *  R8 a row whose length is not a multiple of B ends in a shorter block holding
 *     the remaining elements; it has its own participation bit and is sized like
 *     the others (1 + len*m or 1 + len*w bits).
 */
#include "ibp_oracle.h"

#include <string.h>

#include <vector>

namespace {

/* read element e of a little-endian array of w-bit words */
uint32_t load_elem(const unsigned char *base, int64_t e, int w_bits) {
  int nbytes = w_bits / 8;
  uint32_t v = 0;
  for (int k = 0; k < nbytes; ++k) v |= (uint32_t)base[e * nbytes + k] << (8 * k);
  return v;
}

void store_elem(unsigned char *base, int64_t e, int w_bits, uint32_t v) {
  int nbytes = w_bits / 8;
  for (int k = 0; k < nbytes; ++k) base[e * nbytes + k] = (unsigned char)((v >> (8 * k)) & 0xFFu);
}

int bit_of(uint32_t x, int j) { return (int)((x >> j) & 1u); }

int popcount_w(uint32_t x, int w_bits) {
  int c = 0;
  for (int j = 0; j < w_bits; ++j) c += bit_of(x, j);
  return c;
}

/* the non-invariant bits of x, packed in ascending position order */
uint32_t extract_kept(uint32_t x, uint32_t mask, int w_bits) {
  uint32_t field = 0;
  int k = 0;
  for (int j = 0; j < w_bits; ++j) {
    if (!bit_of(mask, j)) {
      field |= (uint32_t)bit_of(x, j) << k;
      ++k;
    }
  }
  return field;
}

/* inverse of extract_kept: spread field over the non-invariant positions, then
   put the invariant values back */
uint32_t reinsert(uint32_t field, uint32_t mask, uint32_t bitval, int w_bits) {
  uint32_t x = 0;
  int k = 0;
  for (int j = 0; j < w_bits; ++j) {
    if (bit_of(mask, j)) {
      x |= (uint32_t)bit_of(bitval, j) << j;
    } else {
      x |= (uint32_t)bit_of(field, k) << j;
      ++k;
    }
  }
  return x;
}

/* bit stream over little-endian 32-bit words, LSB first */
void put_bit(unsigned char *stream, int64_t pos, int bit) {
  int64_t word = pos / 32;
  int in_word = (int)(pos % 32);
  int64_t byte = word * 4 + in_word / 8;
  int in_byte = in_word % 8;
  if (bit) stream[byte] = (unsigned char)(stream[byte] | (1u << in_byte));
  else stream[byte] = (unsigned char)(stream[byte] & ~(1u << in_byte));
}

int get_bit(const unsigned char *stream, int64_t pos) {
  int64_t word = pos / 32;
  int in_word = (int)(pos % 32);
  int64_t byte = word * 4 + in_word / 8;
  int in_byte = in_word % 8;
  return (stream[byte] >> in_byte) & 1;
}

void put_field(unsigned char *stream, int64_t *pos, uint32_t value, int nbits) {
  for (int i = 0; i < nbits; ++i) {
    put_bit(stream, *pos, bit_of(value, i));
    *pos += 1;
  }
}

uint32_t get_field(const unsigned char *stream, int64_t *pos, int nbits) {
  uint32_t v = 0;
  for (int i = 0; i < nbits; ++i) {
    v |= (uint32_t)get_bit(stream, *pos) << i;
    *pos += 1;
  }
  return v;
}

int valid_width(int w_bits) { return w_bits == 8 || w_bits == 16 || w_bits == 32; }

/* elements of block b of a row: B, except the last block of a row whose length is
   not a multiple of B, which holds the remaining row_elems - b*B (R8) */
int64_t block_len(int64_t b, int64_t row_elems, int64_t block_elems) {
  int64_t end = (b + 1) * block_elems;
  if (end > row_elems) end = row_elems;
  return end - b * block_elems;
}

uint32_t width_mask(int w_bits) { return w_bits == 32 ? 0xFFFFFFFFu : ((1u << w_bits) - 1u); }

}  // namespace

extern "C" int64_t ibpo_slot_bytes(int64_t row_elems, int w_bits) {
  int64_t raw = row_elems * (w_bits / 8);
  return (raw + 15) / 16 * 16;
}

/* Preprocessing: count, per bit position, how many sampled elements hold a 1;
   a position is invariant when its majority value is held by at least a
   fraction T of the sample. */
extern "C" int ibpo_build_meta(const void *elems, int64_t n_elems, int w_bits, double T,
                               uint32_t *mask_out, uint32_t *bitval_out) {
  if (!elems || n_elems <= 0 || !valid_width(w_bits) || !(T >= 0.0 && T <= 1.0) || !mask_out ||
      !bitval_out)
    return IBPO_BAD_ARG;
  const unsigned char *base = (const unsigned char *)elems;
  int64_t ones[32];
  for (int j = 0; j < 32; ++j) ones[j] = 0;
  for (int64_t e = 0; e < n_elems; ++e) {
    uint32_t x = load_elem(base, e, w_bits);
    for (int j = 0; j < w_bits; ++j) ones[j] += bit_of(x, j);
  }
  uint32_t mask = 0, bitval = 0;
  for (int j = 0; j < w_bits; ++j) {
    int64_t c1 = ones[j];
    int64_t c0 = n_elems - c1;
    int v = c1 > c0 ? 1 : 0;               /* R5: a tie picks 0 */
    int64_t cv = v ? c1 : c0;
    if ((double)cv >= T * (double)n_elems) { /* R4 */
      mask |= 1u << j;
      bitval |= (uint32_t)v << j;
    }
  }
  *mask_out = mask;
  *bitval_out = bitval;
  return IBPO_OK;
}

namespace {

/* The code rows are compressed with: for every element position e of a row its
   mask, bitval and field width m. The threshold metadata gives one pair shared by
   all positions; the per-position variant one pair per position. The arrays run
   one block past the row (mask 0, field width w) so that block loops never index
   past them. */
struct PosCode {
  std::vector<uint32_t> mask, bitval;
  std::vector<int> m;
};

PosCode make_code(const uint32_t *pmask, const uint32_t *pbitval, int shared, int64_t row_elems,
                  int64_t block_elems, int w_bits) {
  PosCode c;
  const int64_t n = row_elems + block_elems;
  c.mask.assign((size_t)n, 0u);
  c.bitval.assign((size_t)n, 0u);
  c.m.assign((size_t)n, w_bits);
  for (int64_t e = 0; e < row_elems; ++e) {
    uint32_t mk = (shared ? pmask[0] : pmask[e]) & width_mask(w_bits);
    c.mask[e] = mk;
    c.bitval[e] = (shared ? pbitval[0] : pbitval[e]) & mk;
    c.m[e] = w_bits - popcount_w(mk, w_bits);
  }
  return c;
}

/* payload bits of block b: one field of m_e bits per element when the block
   matches, the raw w-bit words otherwise */
int64_t block_payload_bits(const PosCode &c, int64_t b, int64_t row_elems, int64_t block_elems,
                           int w_bits, int match) {
  const int64_t len = block_len(b, row_elems, block_elems);
  int64_t s = 0;
  for (int64_t i = 0; i < len; ++i) s += match ? c.m[b * block_elems + i] : w_bits;
  return s;
}

/* block b matches when every element holds its position's bitval at its
   position's mask */
int block_matches(const PosCode &c, const unsigned char *row, int64_t b, int64_t row_elems,
                  int64_t block_elems, int w_bits) {
  int match = 1;
  for (int64_t e = b * block_elems; e < b * block_elems + block_len(b, row_elems, block_elems); ++e)
    if ((load_elem(row, e, w_bits) & c.mask[e]) != c.bitval[e]) match = 0;
  return match;
}

/* Compression: test each block against the code, record a participation bit per
   block, strip the invariant bits of matching blocks and close the gaps, keep
   failing blocks as they are; store the row in its fixed-size slot and flag it in
   the bitmask when that saves space. */
int compress_rows(const void *rows, int64_t n_rows, int64_t row_elems, int w_bits,
                  int64_t block_elems, const PosCode &c, void *slots, int64_t slot_bytes,
                  uint32_t *bitmask, uint32_t *row_bits) {
  const unsigned char *in = (const unsigned char *)rows;
  unsigned char *out = (unsigned char *)slots;
  const int64_t raw_bytes = row_elems * (w_bits / 8);
  const int64_t nb = (row_elems + block_elems - 1) / block_elems;

  for (int64_t q = 0; q < (n_rows + 31) / 32; ++q) bitmask[q] = 0;

  for (int64_t r = 0; r < n_rows; ++r) {
    const unsigned char *row = in + r * raw_bytes;
    unsigned char *slot = out + r * slot_bytes;

    /* participation bit per block */
    int64_t bits = 0;
    for (int64_t b = 0; b < nb; ++b) {
      int match = block_matches(c, row, b, row_elems, block_elems, w_bits);
      bits += 1 + block_payload_bits(c, b, row_elems, block_elems, w_bits, match);
    }
    if (row_bits) row_bits[r] = (uint32_t)bits;

    int64_t stored_words = (bits + 31) / 32;
    int compressed = 4 * stored_words < raw_bytes; /* R7 */
    if (!compressed) {
      for (int64_t k = 0; k < raw_bytes; ++k) slot[k] = row[k];
      continue;
    }
    for (int64_t k = 0; k < 4 * stored_words; ++k) slot[k] = 0;
    int64_t pos = 0;
    /* header: all participation bits first (R2) */
    for (int64_t b = 0; b < nb; ++b) {
      put_bit(slot, pos, block_matches(c, row, b, row_elems, block_elems, w_bits));
      pos += 1;
    }
    /* payloads, block by block */
    for (int64_t b = 0; b < nb; ++b) {
      int match = get_bit(slot, b);
      for (int64_t e = b * block_elems; e < b * block_elems + block_len(b, row_elems, block_elems);
           ++e) {
        uint32_t x = load_elem(row, e, w_bits);
        if (match) put_field(slot, &pos, extract_kept(x, c.mask[e], w_bits), c.m[e]);
        else put_field(slot, &pos, x, w_bits);
      }
    }
    bitmask[r / 32] |= 1u << (r % 32);
  }
  return IBPO_OK;
}

}  // namespace

extern "C" int ibpo_compress(const void *rows, int64_t n_rows, int64_t row_elems, int w_bits,
                             int64_t block_elems, uint32_t mask, uint32_t bitval, void *slots,
                             int64_t slot_bytes, uint32_t *bitmask, uint32_t *row_bits) {
  if (!rows || !slots || !bitmask || n_rows < 0 || row_elems <= 0 || !valid_width(w_bits) ||
      block_elems <= 0 || slot_bytes < ibpo_slot_bytes(row_elems, w_bits))
    return IBPO_BAD_ARG;
  const PosCode c = make_code(&mask, &bitval, 1, row_elems, block_elems, w_bits);
  return compress_rows(rows, n_rows, row_elems, w_bits, block_elems, c, slots, slot_bytes,
                       bitmask, row_bits);
}

extern "C" int ibpo_compress_positions(const void *rows, int64_t n_rows, int64_t row_elems,
                                       int w_bits, int64_t block_elems, const uint32_t *pmask,
                                       const uint32_t *pbitval, void *slots, int64_t slot_bytes,
                                       uint32_t *bitmask, uint32_t *row_bits) {
  if (!rows || !slots || !bitmask || !pmask || !pbitval || n_rows < 0 || row_elems <= 0 ||
      !valid_width(w_bits) || block_elems <= 0 || slot_bytes < ibpo_slot_bytes(row_elems, w_bits))
    return IBPO_BAD_ARG;
  const PosCode c = make_code(pmask, pbitval, 0, row_elems, block_elems, w_bits);
  return compress_rows(rows, n_rows, row_elems, w_bits, block_elems, c, slots, slot_bytes,
                       bitmask, row_bits);
}

namespace {

/* Decompression of one row from its stored bytes (slot or packed entry, `avail`
   bytes of it readable): read the participation bits, walk the blocks in order
   (each block's start is the sum of the sizes of the blocks before it), and
   rebuild every element by putting the invariant bits back in place. Returns
   IBPO_OK, or IBPO_CORRUPT (orow untouched) when the stream the participation bits
   describe would not have been stored compressed or does not fit `avail`. */
int decode_row(const unsigned char *slot, int64_t avail, int compressed, int64_t row_elems,
               int w_bits, int64_t block_elems, const PosCode &c, unsigned char *orow) {
  const int64_t raw_bytes = row_elems * (w_bits / 8);
  const int64_t nb = (row_elems + block_elems - 1) / block_elems;
  if (!compressed) {
    if (avail < raw_bytes) return IBPO_CORRUPT;
    for (int64_t k = 0; k < raw_bytes; ++k) orow[k] = slot[k];
    return IBPO_OK;
  }
  if (avail * 8 < nb) return IBPO_CORRUPT;
  int64_t bits = 0;
  for (int64_t b = 0; b < nb; ++b)
    bits += 1 + block_payload_bits(c, b, row_elems, block_elems, w_bits, get_bit(slot, b));
  if (4 * ((bits + 31) / 32) >= raw_bytes || 4 * ((bits + 31) / 32) > avail) return IBPO_CORRUPT;
  int64_t pos = nb; /* first payload bit */
  for (int64_t b = 0; b < nb; ++b) {
    int match = get_bit(slot, b);
    for (int64_t e = b * block_elems; e < b * block_elems + block_len(b, row_elems, block_elems);
         ++e) {
      uint32_t x;
      if (match) x = reinsert(get_field(slot, &pos, c.m[e]), c.mask[e], c.bitval[e], w_bits);
      else x = get_field(slot, &pos, w_bits);
      store_elem(orow, e, w_bits, x);
    }
  }
  return IBPO_OK;
}

int gather_rows(const void *slots, int64_t slot_bytes, int64_t n_rows, int64_t row_elems,
                int w_bits, int64_t block_elems, const uint32_t *bitmask, const PosCode &c,
                const int64_t *idx, int64_t n_idx, void *out) {
  const unsigned char *in = (const unsigned char *)slots;
  unsigned char *dst = (unsigned char *)out;
  const int64_t raw_bytes = row_elems * (w_bits / 8);
  int status = IBPO_OK;
  for (int64_t i = 0; i < n_idx; ++i) {
    int64_t r = idx[i];
    if (r < 0 || r >= n_rows) {
      if (status == IBPO_OK) status = IBPO_BAD_INDEX;
      continue;
    }
    int compressed = (int)((bitmask[r / 32] >> (r % 32)) & 1u);
    int rc = decode_row(in + r * slot_bytes, slot_bytes, compressed, row_elems, w_bits,
                        block_elems, c, dst + i * raw_bytes);
    if (rc != IBPO_OK && status == IBPO_OK) status = rc;
  }
  return status;
}

}  // namespace

/* Decompression-gather: rebuild each requested row from its slot. */
extern "C" int ibpo_decompress_gather(const void *slots, int64_t slot_bytes, int64_t n_rows,
                                      int64_t row_elems, int w_bits, int64_t block_elems,
                                      const uint32_t *bitmask, uint32_t mask, uint32_t bitval,
                                      const int64_t *idx, int64_t n_idx, void *out) {
  if (n_idx < 0 || n_rows < 0 || row_elems <= 0 || !valid_width(w_bits) || block_elems <= 0 ||
      slot_bytes < ibpo_slot_bytes(row_elems, w_bits))
    return IBPO_BAD_ARG;
  if (n_idx == 0) return IBPO_OK;
  if (!slots || !bitmask || !idx || !out) return IBPO_BAD_ARG;
  const PosCode c = make_code(&mask, &bitval, 1, row_elems, block_elems, w_bits);
  return gather_rows(slots, slot_bytes, n_rows, row_elems, w_bits, block_elems, bitmask, c, idx,
                     n_idx, out);
}

extern "C" int ibpo_decompress_gather_positions(const void *slots, int64_t slot_bytes,
                                                int64_t n_rows, int64_t row_elems, int w_bits,
                                                int64_t block_elems, const uint32_t *bitmask,
                                                const uint32_t *pmask, const uint32_t *pbitval,
                                                const int64_t *idx, int64_t n_idx, void *out) {
  if (n_idx < 0 || n_rows < 0 || row_elems <= 0 || !valid_width(w_bits) || block_elems <= 0 ||
      slot_bytes < ibpo_slot_bytes(row_elems, w_bits))
    return IBPO_BAD_ARG;
  if (n_idx == 0) return IBPO_OK;
  if (!slots || !bitmask || !idx || !out || !pmask || !pbitval) return IBPO_BAD_ARG;
  const PosCode c = make_code(pmask, pbitval, 0, row_elems, block_elems, w_bits);
  return gather_rows(slots, slot_bytes, n_rows, row_elems, w_bits, block_elems, bitmask, c, idx,
                     n_idx, out);
}

/* Per-position metadata: the preprocessing rule applied to each element position
   of a row on its own (the sample of position e is element e of every row). */
extern "C" int ibpo_build_meta_positions(const void *rows, int64_t n_rows, int64_t row_elems,
                                         int w_bits, double T, uint32_t *pmask_out,
                                         uint32_t *pbitval_out) {
  if (!rows || n_rows <= 0 || row_elems <= 0 || !valid_width(w_bits) || !pmask_out ||
      !pbitval_out)
    return IBPO_BAD_ARG;
  const unsigned char *base = (const unsigned char *)rows;
  const int nbytes = w_bits / 8;
  std::vector<unsigned char> column((size_t)(n_rows * nbytes));
  for (int64_t e = 0; e < row_elems; ++e) {
    for (int64_t r = 0; r < n_rows; ++r)
      for (int k = 0; k < nbytes; ++k)
        column[(size_t)(r * nbytes + k)] = base[(r * row_elems + e) * nbytes + k];
    int rc = ibpo_build_meta(column.data(), n_rows, w_bits, T, &pmask_out[e], &pbitval_out[e]);
    if (rc != IBPO_OK) return rc;
  }
  return IBPO_OK;
}

/* Block-position metadata: one mask/bitval per position q within a block, from the
 * sample made of the element at position q of every block of every row (a shorter
 * last block adds only the positions it has); element e of a row takes the pair of
 * its position e % block_elems. */
extern "C" int ibpo_build_meta_block_positions(const void *rows, int64_t n_rows,
                                               int64_t row_elems, int w_bits, double T,
                                               int64_t block_elems, uint32_t *pmask_out,
                                               uint32_t *pbitval_out) {
  if (!rows || n_rows <= 0 || row_elems <= 0 || block_elems <= 0 || !valid_width(w_bits) ||
      !pmask_out || !pbitval_out)
    return IBPO_BAD_ARG;
  const unsigned char *base = (const unsigned char *)rows;
  const int nbytes = w_bits / 8;
  const int64_t npos = block_elems < row_elems ? block_elems : row_elems;
  std::vector<unsigned char> sample;
  for (int64_t q = 0; q < npos; ++q) {
    sample.clear();
    for (int64_t r = 0; r < n_rows; ++r)
      for (int64_t e = q; e < row_elems; e += block_elems)
        for (int k = 0; k < nbytes; ++k) sample.push_back(base[(r * row_elems + e) * nbytes + k]);
    uint32_t mask = 0, bitval = 0;
    int rc = ibpo_build_meta(sample.data(), (int64_t)(sample.size() / nbytes), w_bits, T, &mask,
                             &bitval);
    if (rc != IBPO_OK) return rc;
    for (int64_t e = q; e < row_elems; e += block_elems) {
      pmask_out[e] = mask;
      pbitval_out[e] = bitval;
    }
  }
  return IBPO_OK;
}

/* Packed store: each selected row's used bytes, rounded up to 16, end to end. */
extern "C" int ibpo_pack(const void *slots, int64_t slot_bytes, int64_t n_rows, int64_t row_elems,
                         int w_bits, const uint32_t *bitmask, const uint32_t *row_bits,
                         const int64_t *sel, int64_t n_sel, int64_t *offsets, void *packed,
                         uint32_t *pack_bitmask, uint32_t *pack_row_bits) {
  if (!slots || !bitmask || !row_bits || !offsets || n_rows < 0 || n_sel < 0 || row_elems <= 0 ||
      !valid_width(w_bits) || slot_bytes < ibpo_slot_bytes(row_elems, w_bits) ||
      (!sel && n_sel > n_rows))
    return IBPO_BAD_ARG;
  const unsigned char *in = (const unsigned char *)slots;
  unsigned char *out = (unsigned char *)packed;
  const int64_t raw_bytes = row_elems * (w_bits / 8);
  if (packed && pack_bitmask)
    for (int64_t q = 0; q < (n_sel + 31) / 32; ++q) pack_bitmask[q] = 0;
  int64_t at = 0;
  for (int64_t i = 0; i < n_sel; ++i) {
    int64_t r = sel ? sel[i] : i;
    if (r < 0 || r >= n_rows) return IBPO_BAD_INDEX;
    int compressed = (int)((bitmask[r / 32] >> (r % 32)) & 1u);
    int64_t used = compressed ? 4 * (((int64_t)row_bits[r] + 31) / 32) : raw_bytes;
    int64_t len = (used + 15) / 16 * 16;
    offsets[i] = at;
    if (packed) {
      for (int64_t k = 0; k < len; ++k) out[at + k] = in[r * slot_bytes + k];
      if (pack_bitmask && compressed) pack_bitmask[i / 32] |= 1u << (i % 32);
      if (pack_row_bits) pack_row_bits[i] = row_bits[r];
    }
    at += len;
  }
  offsets[n_sel] = at;
  return IBPO_OK;
}

/* Decompression-gather from a packed store. */
extern "C" int ibpo_decompress_gather_packed(const void *packed, const int64_t *offsets,
                                             int64_t n_rows, int64_t row_elems, int w_bits,
                                             int64_t block_elems, const uint32_t *bitmask,
                                             uint32_t mask, uint32_t bitval, const int64_t *idx,
                                             int64_t n_idx, void *out) {
  if (n_idx < 0 || n_rows < 0 || row_elems <= 0 || !valid_width(w_bits) || block_elems <= 0)
    return IBPO_BAD_ARG;
  if (n_idx == 0) return IBPO_OK;
  if (!packed || !offsets || !bitmask || !idx || !out) return IBPO_BAD_ARG;
  const PosCode c = make_code(&mask, &bitval, 1, row_elems, block_elems, w_bits);
  const unsigned char *in = (const unsigned char *)packed;
  unsigned char *dst = (unsigned char *)out;
  const int64_t raw_bytes = row_elems * (w_bits / 8);
  int status = IBPO_OK;
  for (int64_t i = 0; i < n_idx; ++i) {
    int64_t r = idx[i];
    if (r < 0 || r >= n_rows) {
      if (status == IBPO_OK) status = IBPO_BAD_INDEX;
      continue;
    }
    int compressed = (int)((bitmask[r / 32] >> (r % 32)) & 1u);
    int64_t avail = offsets[r + 1] - offsets[r];
    int rc = avail < 0 ? IBPO_CORRUPT
                       : decode_row(in + offsets[r], avail, compressed, row_elems, w_bits,
                                    block_elems, c, dst + i * raw_bytes);
    if (rc != IBPO_OK && status == IBPO_OK) status = rc;
  }
  return status;
}

/* Saving-aware mask selection: start from the threshold rule's mask and drop
   its least-held positions one group at a time; compress the rows under every
   mask so obtained and keep the one that stores them in the fewest bytes. */
extern "C" int ibpo_select_meta(const void *rows, int64_t n_rows, int64_t row_elems, int w_bits,
                                double T, int64_t block_elems, uint32_t *mask_out,
                                uint32_t *bitval_out, uint32_t *cand_mask, int64_t *cand_bytes,
                                int *n_cand) {
  if (!rows || n_rows <= 0 || row_elems <= 0 || !valid_width(w_bits) || block_elems <= 0 ||
      !(T >= 0.0 && T <= 1.0) || !mask_out || !bitval_out)
    return IBPO_BAD_ARG;
  const int64_t n_elems = n_rows * row_elems;
  uint32_t mask0 = 0, bitval0 = 0;
  if (ibpo_build_meta(rows, n_elems, w_bits, T, &mask0, &bitval0) != IBPO_OK) return IBPO_BAD_ARG;

  /* how many elements hold the majority value of each position */
  const unsigned char *base = (const unsigned char *)rows;
  int64_t ones[32];
  for (int j = 0; j < 32; ++j) ones[j] = 0;
  for (int64_t e = 0; e < n_elems; ++e) {
    uint32_t x = load_elem(base, e, w_bits);
    for (int j = 0; j < w_bits; ++j) ones[j] += bit_of(x, j);
  }
  int64_t held[32];
  for (int j = 0; j < w_bits; ++j) {
    int64_t c1 = ones[j], c0 = n_elems - c1;
    held[j] = c1 > c0 ? c1 : c0;
  }

  /* the candidate masks, largest first */
  std::vector<uint32_t> cands;
  uint32_t cur = mask0;
  cands.push_back(cur);
  while (cur != 0) {
    int64_t fewest = -1;
    for (int j = 0; j < w_bits; ++j)
      if (bit_of(cur, j) && (fewest < 0 || held[j] < fewest)) fewest = held[j];
    for (int j = 0; j < w_bits; ++j)
      if (bit_of(cur, j) && held[j] == fewest) cur &= ~(1u << j);
    cands.push_back(cur);
  }

  /* score each by compressing every row with it */
  const int64_t raw_bytes = row_elems * (w_bits / 8);
  const int64_t sb = ibpo_slot_bytes(row_elems, w_bits);
  std::vector<unsigned char> slots((size_t)(n_rows * sb));
  std::vector<uint32_t> bitmask((size_t)((n_rows + 31) / 32));
  std::vector<uint32_t> row_bits((size_t)n_rows);
  std::vector<int64_t> total(cands.size());
  for (size_t k = 0; k < cands.size(); ++k) {
    uint32_t mk = cands[k], bk = bitval0 & cands[k];
    if (ibpo_compress(rows, n_rows, row_elems, w_bits, block_elems, mk, bk, slots.data(), sb,
                      bitmask.data(), row_bits.data()) != IBPO_OK)
      return IBPO_BAD_ARG;
    int64_t sum = 0;
    for (int64_t r = 0; r < n_rows; ++r) {
      int compressed = (int)((bitmask[r / 32] >> (r % 32)) & 1u);
      sum += compressed ? 4 * (((int64_t)row_bits[r] + 31) / 32) : raw_bytes;
    }
    total[k] = sum;
  }
  size_t best = 0;
  for (size_t k = 1; k < cands.size(); ++k)
    if (total[k] < total[best]) best = k; /* strict: ties keep the larger mask */

  *mask_out = cands[best];
  *bitval_out = bitval0 & cands[best];
  if (cand_mask && cand_bytes) {
    for (int k = 0; k < 33; ++k) {
      cand_mask[k] = k < (int)cands.size() ? cands[k] : 0u;
      cand_bytes[k] = k < (int)cands.size() ? total[k] : -1;
    }
  }
  if (n_cand) *n_cand = (int)cands.size();
  return IBPO_OK;
}
