/*
 * Plain single-threaded CPU oracle for Invariant Bit Packing (IBP).
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check of the package
 * entry file and the CPU-baseline leg of the benchmark may load this library.
 * The GPU codec never links, calls or includes anything from this directory,
 * and this directory includes nothing from the GPU codec.
 *
 * Source of the method: "Reducing the GPU Memory Bottleneck with Lossless
 * Compression for ML -- Extended" (Kamath, Krishnamurthy, Canini, Peter),
 * technical summary, sections "Core algorithm" (preprocessing / compression /
 * decompression) and "System integration" (PCIe transfer compression with
 * fixed-size buffers and a GPU-resident bitmask).
 *
 * Every routine works on bit patterns only: elements are w-bit little-endian
 * words (w = 32 for FP32, 16 for FP16/BF16); no floating-point value is ever
 * interpreted, so +-0, denormals, Inf and NaN payloads are ordinary words.
 *
 * Stream format (the pages leave it open; the readings are listed in the design
 * notes and repeated in the .cpp):
 *   - a row of L elements is cut into nb = L/B blocks of B elements;
 *   - participation bit p_b = 1 iff every element x of block b satisfies
 *     (x & mask) == bitval;
 *   - the row's bit stream is: nb participation bits (bit b = p_b), then for each
 *     block in order either B fields of m = w - popcount(mask) bits (the element's
 *     non-invariant bits in ascending position order) when p_b = 1, or B raw
 *     w-bit words when p_b = 0;
 *   - stream bit i is bit (i mod 32) of little-endian 32-bit word i/32;
 *   - the row is stored compressed iff 4*ceil(bits/32) < L*w/8; then its slot
 *     holds the stream (zero padded to the end of the last used word) and row
 *     bit r of the bitmask is 1; otherwise the slot holds the raw row and the
 *     bitmask bit is 0.
 */
#ifndef IBP_ORACLE_H
#define IBP_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes of the oracle (its own numbering) */
#define IBPO_OK 0
#define IBPO_BAD_ARG (-1)
#define IBPO_BAD_INDEX (-5)
#define IBPO_CORRUPT (-6)

/* Metadata (technical summary, core algorithm: preprocessing).
 * elems: n_elems little-endian words of w_bits (16 or 32) bits.
 * For each bit position j < w: c1 = number of elements whose bit j is 1,
 * c0 = n_elems - c1; the majority value v = (c1 > c0); bit j is invariant iff
 * (double)count_of_v >= T * (double)n_elems. Writes mask (invariant positions)
 * and bitval (their values; zero outside mask). Returns IBPO_OK or IBPO_BAD_ARG. */
int ibpo_build_meta(const void *elems, int64_t n_elems, int w_bits, double T,
                    uint32_t *mask_out, uint32_t *bitval_out);

/* Per-position metadata (a variant of preprocessing: the "kilobyte-scale"
 * metadata reading). Element position e of a row (0 <= e < row_elems) gets its own
 * mask/bitval pair: the preprocessing rule of ibpo_build_meta applied to the
 * sample made of element e of every row. pmask_out/pbitval_out: row_elems words. */
int ibpo_build_meta_positions(const void *rows, int64_t n_rows, int64_t row_elems, int w_bits,
                              double T, uint32_t *pmask_out, uint32_t *pbitval_out);

/* Block-position metadata (a variant of preprocessing: the block-sized reading of the
 * "kilobyte-scale" metadata). Position q of a block (0 <= q < block_elems) gets its
 * own mask/bitval pair: the rule of ibpo_build_meta applied to the sample made of
 * the element at position q of every block of every row (a shorter last block adds
 * only the positions it has). Written row-sized, like ibpo_build_meta_positions:
 * element e of a row gets the pair of position e % block_elems, so the per-position
 * compression and gather take the result as it is. */
int ibpo_build_meta_block_positions(const void *rows, int64_t n_rows, int64_t row_elems,
                                    int w_bits, double T, int64_t block_elems,
                                    uint32_t *pmask_out, uint32_t *pbitval_out);

/* Compression and decompress-gather with per-position metadata: as ibpo_compress /
 * ibpo_decompress_gather, except that element e of a block is tested against
 * pmask[e]/pbitval[e] and, in a matching block, stored as a field of
 * w - popcount(pmask[e]) bits (its non-invariant bits in ascending order). */
int ibpo_compress_positions(const void *rows, int64_t n_rows, int64_t row_elems, int w_bits,
                            int64_t block_elems, const uint32_t *pmask, const uint32_t *pbitval,
                            void *slots, int64_t slot_bytes, uint32_t *bitmask,
                            uint32_t *row_bits);
int ibpo_decompress_gather_positions(const void *slots, int64_t slot_bytes, int64_t n_rows,
                                     int64_t row_elems, int w_bits, int64_t block_elems,
                                     const uint32_t *bitmask, const uint32_t *pmask,
                                     const uint32_t *pbitval, const int64_t *idx, int64_t n_idx,
                                     void *out);

/* Packed store (technical summary, "System integration": the compressed GPU
 * cache that raises the cache's effective capacity). Rows sel[0..n_sel) of a
 * slotted store (sel == NULL: rows 0..n_sel) are laid end to end: entry i holds the
 * used prefix of slot sel[i] (4*ceil(bits/32) bytes for a compressed row, the raw
 * row otherwise) rounded up to a multiple of 16 bytes (bytes copied from the slot).
 * offsets[i] = byte offset of entry i; offsets[n_sel] = total bytes (n_sel + 1
 * entries). pack_bitmask bit i / pack_row_bits[i] = the source row's bitmask bit
 * and bit count. packed may be NULL to compute only the offsets. Returns IBPO_OK,
 * IBPO_BAD_ARG, or IBPO_BAD_INDEX for a selection outside [0, n_rows). */
int ibpo_pack(const void *slots, int64_t slot_bytes, int64_t n_rows, int64_t row_elems,
              int w_bits, const uint32_t *bitmask, const uint32_t *row_bits, const int64_t *sel,
              int64_t n_sel, int64_t *offsets, void *packed, uint32_t *pack_bitmask,
              uint32_t *pack_row_bits);

/* Decompress-gather from a packed store: as ibpo_decompress_gather, with row r's
 * bytes at packed + offsets[r] and offsets[r+1] - offsets[r] of them; a row whose
 * stream (or raw row) does not fit its entry is treated as corrupt. */
int ibpo_decompress_gather_packed(const void *packed, const int64_t *offsets, int64_t n_rows,
                                  int64_t row_elems, int w_bits, int64_t block_elems,
                                  const uint32_t *bitmask, uint32_t mask, uint32_t bitval,
                                  const int64_t *idx, int64_t n_idx, void *out);

/* Saving-aware mask selection (a variant of preprocessing that trades some
 * invariant positions for more matching blocks; the threshold rule alone can keep
 * a position whose rare exceptions spoil most blocks).
 * Candidates: candidate 0 is the threshold rule's mask M0 (ibpo_build_meta over
 * all n_rows*row_elems elements); candidate k+1 is candidate k without the
 * positions, among those it still holds, whose majority value is held by the
 * fewest elements (positions with equal counts leave together); the last
 * candidate is the empty mask. Each candidate's bitval is M0's bitval restricted
 * to it. Each candidate is scored by compressing all rows with it (ibpo_compress)
 * and summing the bytes each row occupies (4*ceil(bits/32) when compressed, else
 * the raw row); the smallest sum wins, ties going to the lower k (the larger mask).
 * Writes the winner to mask_out/bitval_out; when cand_mask/cand_bytes are not
 * null (33 entries each) writes every candidate's mask and byte total and
 * *n_cand = number of candidates (1..w+1). Returns IBPO_OK or IBPO_BAD_ARG. */
int ibpo_select_meta(const void *rows, int64_t n_rows, int64_t row_elems, int w_bits, double T,
                     int64_t block_elems, uint32_t *mask_out, uint32_t *bitval_out,
                     uint32_t *cand_mask, int64_t *cand_bytes, int *n_cand);

/* Slot size for a row: raw bytes L*w/8 rounded up to a multiple of 16. */
int64_t ibpo_slot_bytes(int64_t row_elems, int w_bits);

/* Compression (technical summary, core algorithm: compression; system
 * integration: fixed-size buffers + bitmask). rows: n_rows x row_elems words.
 * slots: n_rows x slot_bytes bytes (every byte of a used slot prefix is written;
 * for compressed rows bytes past the last used word are left untouched).
 * bitmask: ceil(n_rows/32) words, fully rewritten (bits past n_rows = 0).
 * row_bits (nullable): per-row sum over blocks of (1 + B*m) or (1 + B*w). */
int ibpo_compress(const void *rows, int64_t n_rows, int64_t row_elems, int w_bits,
                  int64_t block_elems, uint32_t mask, uint32_t bitval, void *slots,
                  int64_t slot_bytes, uint32_t *bitmask, uint32_t *row_bits);

/* Decompress-gather (technical summary, core algorithm: decompression).
 * out[i] = original row idx[i], for i < n_idx. An index outside [0, n_rows)
 * leaves out[i] untouched and makes the call return IBPO_BAD_INDEX; a compressed
 * slot whose participation bits describe a stream of at least the raw size leaves
 * out[i] untouched and makes the call return IBPO_CORRUPT (first error wins). */
int ibpo_decompress_gather(const void *slots, int64_t slot_bytes, int64_t n_rows,
                           int64_t row_elems, int w_bits, int64_t block_elems,
                           const uint32_t *bitmask, uint32_t mask, uint32_t bitval,
                           const int64_t *idx, int64_t n_idx, void *out);

#ifdef __cplusplus
}
#endif
#endif
