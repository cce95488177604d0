/*
 * ibp.h -- C ABI of the GB300 (sm_103a) Invariant Bit Packing codec.
 *
 * Method: "Reducing the GPU Memory Bottleneck with Lossless Compression for ML --
 * Extended" (Kamath, Krishnamurthy, Canini, Peter), technical summary:
 *   - "Core algorithm", preprocessing: find the bit positions of the element word
 *     that hold one value in at least a fraction T of a sample, keep them as a
 *     fixed-size mask + bitval in GPU memory, reuse them for the whole dataset;
 *   - "Core algorithm", compression: per fixed-size block, test the invariant
 *     positions against bitval; on a match strip them and close the gaps; mark
 *     each block with a participation bit; run on the GPU over zero-copy memory;
 *   - "Core algorithm", decompression: a warp stages a contiguous compressed
 *     segment in shared memory, prefix-scans block sizes with warp primitives to
 *     find each block's bit offset, and reinserts the invariant bits;
 *   - "System integration", PCIe transfer compression: one fixed-size buffer per
 *     tensor of which only the compressed part is read, plus a GPU-resident
 *     bitmask of which tensors are compressed.
 *
 * Conventions shared by every call
 *   - A "row" is the unit stored in one slot (a feature vector, an embedding
 *     row, a weight row, a token's K or V). Rows are row_elems little-endian
 *     element words of w bits: w = 32 (IBP_FP32), 16 (IBP_FP16, IBP_BF16) or 8
 *     (IBP_W8).
 *     Only bit patterns are handled: +-0, denormals, Inf and NaN payloads are
 *     ordinary words and always round-trip exactly.
 *   - block_elems B must be 32 or 64; 1 <= row_elems <= 2^20. A row is cut into
 *     nb = ceil(row_elems / B) blocks; when B does not divide row_elems the last
 *     block holds the remaining elements (its own participation bit, sized
 *     1 + len*m or 1 + len*w bits), and the row must then be a multiple of 16
 *     bytes long (row_elems * w / 8 % 16 == 0).
 *   - Slot r of a store starts at slots + r*slot_bytes; slot_bytes is at least
 *     ibp_slot_bytes() (the raw row rounded up to 16 bytes) and a multiple of 16.
 *   - Stream format of a compressed row (bit i = bit i%32 of little-endian 32-bit
 *     word i/32): nb participation bits, then each block in order, either one
 *     field of m = w - popcount(mask) bits per element (the element's
 *     non-invariant bits, ascending) or the raw words. A row is stored compressed
 *     iff 4*ceil(bits/32) < raw bytes, where bits = sum_b (1 + len_b*m) or
 *     (1 + len_b*w), len_b = B except for a shorter last block.
 *   - Bitmask: bit r of a store is bit r%32 of 32-bit word r/32.
 *   - Ownership: the caller owns and allocates every buffer; the library
 *     allocates nothing, keeps no per-call state and never synchronises a stream
 *     except where stated. Pointers named d_* must be device memory. rows and
 *     slots may be device memory or page-locked host memory registered with CUDA
 *     (read and written zero-copy by the kernels); pageable host memory is
 *     rejected. rows, slots and out must be 16-byte aligned.
 *   - Every compute call is asynchronous on stream s (0 = legacy default stream)
 *     and may be captured in a CUDA graph once the argument checks pass.
 *
 * Return codes: IBP_OK (0) or a negative code found before anything is launched.
 * Errors a kernel detects are written to *d_status (when it is non-null) with an
 * atomic compare-and-swap from 0, so the first error wins; the caller zeroes
 * *d_status before the call. No kernel traps, asserts or waits without bound.
 */
#ifndef IBP_H
#define IBP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *ibp_stream_t; /* same object as cudaStream_t */

/* Element word widths: 32 bits (FP32), 16 bits (FP16, BF16), 8 bits (IBP_W8: FP8
 * E4M3/E5M2, int8, uint8 -- only the width matters, bit patterns are opaque). */
typedef enum { IBP_FP32 = 0, IBP_FP16 = 1, IBP_BF16 = 2, IBP_W8 = 3 } ibp_dtype;

enum {
  IBP_OK = 0,
  IBP_ERR_ARG = -1,         /* null/misaligned/pageable pointer, bad size, T outside [0,1] */
  IBP_ERR_DTYPE = -2,       /* dtype not one of ibp_dtype */
  IBP_ERR_UNSUPPORTED = -3, /* block size or row length the kernels do not handle */
  IBP_ERR_CUDA = -4,        /* a CUDA call or launch failed */
  IBP_ERR_INDEX = -5,       /* (device) gather index outside [0, n_rows) */
  IBP_ERR_CORRUPT = -6,     /* (device) participation bits describe an impossible stream */
  IBP_ERR_META = -7,        /* (device) *d_meta disagrees with the dtype/block_elems passed */
  IBP_ERR_TIMEOUT = -8      /* (device) a bounded wait inside a kernel ran out; output incomplete */
};

/* Metadata: the fixed-size mask/bitval pair of the preprocessing stage.
 * Plain data (16 bytes); the caller may copy or serialise it. mask has a 1 at
 * every invariant bit position; bitval holds their values and is 0 elsewhere.
 * dtype == IBP_META_INVALID marks metadata that ibp_meta_finalize refused to build
 * (every call given it reports IBP_ERR_META). */
#define IBP_META_INVALID 0xFFFFFFFFu

typedef struct {
  uint32_t mask;
  uint32_t bitval;
  uint32_t dtype;       /* ibp_dtype */
  uint32_t block_elems; /* B */
} ibp_meta;

/* Store statistics written by ibp_query / ibp_query_async. */
typedef struct {
  int64_t n_rows;
  int64_t n_compressed; /* rows whose bitmask bit is 1 */
  int64_t raw_bytes;    /* n_rows * row_elems * w/8 */
  int64_t stored_bytes; /* sum over rows: 4*ceil(bits/32) if compressed, else raw row bytes */
  int64_t total_bits;   /* sum over rows of the size formula, compressed or not */
} ibp_stats;

/* Human-readable name of a return/status code (static string). */
const char *ibp_status_string(int code);

/* Bytes of one slot ("System integration": every tensor gets one fixed-size buffer
 * whose leading, compressed part is all that is read; the buffer must hold the row
 * raw, since a row that does not shrink is stored as it is): row_elems * w/8
 * rounded up to 16 (the kernels move 16-byte vectors). row_elems <= 0: IBP_ERR_ARG;
 * unknown dtype: IBP_ERR_DTYPE. Pure host arithmetic, no CUDA call. */
int ibp_slot_bytes(int64_t row_elems, int dtype, int64_t *slot_bytes);

/* Bytes of device scratch ibp_build_meta needs ("Core algorithm", preprocessing:
 * the metadata follows from how often each bit position of the element word holds
 * a 1 in the sample, so the scratch holds one 64-bit count per bit position of a
 * 32-bit word: 256 bytes, whatever the input size). Host arithmetic only. */
int ibp_meta_scratch_bytes(size_t *bytes);

/* Preprocessing ("Core algorithm", preprocessing).
 * rows: n_rows x row_elems element words (device or registered host memory).
 * For every bit position j < w, counts the sampled elements whose bit j is 1; j is
 * invariant iff the majority value's count c satisfies (double)c >= T*(double)N in
 * IEEE double (N = n_rows*row_elems; a tie counts as majority value 0).
 * Writes *d_meta = {mask, bitval, dtype, block_elems}. d_scratch: device memory of
 * ibp_meta_scratch_bytes(), overwritten (no initial contents needed). */
int ibp_build_meta(const void *rows, int64_t n_rows, int64_t row_elems, int dtype, double T,
                   uint32_t block_elems, ibp_meta *d_meta, void *d_scratch, ibp_stream_t s);

/* Preprocessing ("Core algorithm", preprocessing) in two steps, for rows held in
 * several places (shards of a table on several GPUs, or batches streamed one after
 * another): the per-position counts of disjoint row sets add up.
 * ibp_meta_count: rows as for ibp_build_meta (device or registered host memory, a
 * whole number of 32-bit words, 16-byte aligned; n_rows may be 0). Overwrites
 * d_counters (32 uint64 words = 256 bytes of device memory, 8-byte aligned) with the
 * number of 1s at each bit position of the rows' 32-bit words (8- and 16-bit elements
 * are folded into their element positions by the finalize step).
 * The holders' counters are then summed by the caller (an all-reduce of the 32 words
 * across GPUs, or an elementwise add on one GPU).
 * ibp_meta_finalize: applies the threshold rule of ibp_build_meta to the summed
 * counters, n_elems (> 0) being the total number of elements counted, and writes
 * *d_meta. T outside [0, 1] or n_elems <= 0: IBP_ERR_ARG; block_elems not 32 or 64:
 * IBP_ERR_UNSUPPORTED. A counter larger than n_elems (the counters and the element
 * count do not describe the same rows, e.g. one holder's count passed with summed
 * counters) is detected on the device: *d_meta is then written with mask = bitval =
 * 0 and dtype = IBP_META_INVALID, so that every later call given it reports
 * IBP_ERR_META, and IBP_ERR_META is recorded in *d_status (nullable, device memory,
 * compare-and-swap from 0). With one holder the pair equals ibp_build_meta. Both
 * calls are asynchronous on s and allocate nothing. */
int ibp_meta_count(const void *rows, int64_t n_rows, int64_t row_elems, int dtype,
                   uint64_t *d_counters, ibp_stream_t s);
int ibp_meta_finalize(const uint64_t *d_counters, int64_t n_elems, int dtype, double T,
                      uint32_t block_elems, ibp_meta *d_meta, int32_t *d_status,
                      ibp_stream_t s);

/* ibp_build_meta for callers that cannot allocate device memory (the paper has no
 * counterpart; this is a library convenience). Same arguments, checks and result
 * as ibp_build_meta, except that the counters live in a 256-byte array built into
 * the library (kept by every GPU that loads it until the process exits) instead of
 * caller-provided scratch. Meant for code that must not call cudaMalloc when it
 * needs the metadata: a plug-in inside a framework whose allocator owns all device
 * memory, a latency-critical loop where an allocation's implicit synchronisation is
 * not allowed, a system that forbids allocation after start-up.
 * - Allocates nothing: no cudaMalloc/cudaFree and no allocating library call.
 * - The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture. The address is kept together with the identity of the CUDA context it
 *   was looked up in; after a device reset (a new primary context, where the
 *   library's device code is loaded again) the next call looks it up again, so
 *   make that call, too, before any capture.
 * - The counters are cleared on stream s at the start of every call, so results
 *   never depend on an earlier call; but every call shares the one array, so calls
 *   whose kernels overlap on the GPU (e.g. on unordered streams) race and give
 *   undefined results. Order them on one stream or with events.
 * - Returns IBP_ERR_UNSUPPORTED if the counters ever needed more than the 256 bytes
 *   built in (ibp_meta_scratch_bytes() is 256 for every input size today). */
int ibp_build_meta_noalloc(const void *rows, int64_t n_rows, int64_t row_elems, int dtype,
                           double T, uint32_t block_elems, ibp_meta *d_meta, ibp_stream_t s);

/* Saving-aware metadata: a variant of preprocessing (the paper has no counterpart;
 * it follows from "Core algorithm": the threshold rule picks positions one by one,
 * but compression strips a block's invariant bits only when every one of them
 * holds in every element, so a position whose few exceptions fall in many blocks
 * can cost more than it saves).
 * Candidates: candidate 0 is the mask ibp_build_meta gives for T (M0); candidate
 * k+1 is candidate k without every position whose majority value is held by the
 * fewest elements among the positions candidate k still has (equal counts leave
 * together); the last candidate is the empty mask, so there are 1 to w+1 of them.
 * Each candidate's bitval is M0's bitval restricted to it. Each candidate is scored
 * by the bytes rows [0, n_rows) take when compressed with it: the sum over rows of
 * 4*ceil(bits/32) for a row stored compressed and the raw row bytes otherwise.
 * *d_meta receives the lowest-scoring candidate, ties going to the lower k (the
 * larger mask). With T <= 0.5 every position is in M0 and the candidates are all
 * the masks the threshold rule gives for any threshold, plus the empty mask.
 * d_candidates (nullable; device memory of IBP_MAX_MASK_CANDIDATES entries): entry
 * k receives candidate k and its score; entries past the last candidate receive
 * mask = bitval = 0 and stored_bytes = -1.
 * d_scratch: ibp_meta_select_scratch_bytes() bytes of device memory, overwritten.
 * Reads the rows twice (counting, then scoring); same argument checks and codes as
 * ibp_build_meta. */
#define IBP_MAX_MASK_CANDIDATES 33

typedef struct {
  uint32_t mask;
  uint32_t bitval;
  int64_t stored_bytes; /* score of this candidate, or -1 for an unused entry */
} ibp_mask_candidate;   /* 16 bytes */

int ibp_meta_select_scratch_bytes(size_t *bytes);

int ibp_build_meta_select(const void *rows, int64_t n_rows, int64_t row_elems, int dtype,
                          double T, uint32_t block_elems, ibp_meta *d_meta,
                          ibp_mask_candidate *d_candidates, void *d_scratch, ibp_stream_t s);

/* Compression ("Core algorithm", compression; "System integration").
 * Encodes rows [0, n_rows) into their slots with the mask/bitval in *d_meta, whose
 * dtype and block_elems must equal the ones passed. Compressed rows hold their
 * stream in the first 4*ceil(bits/32) bytes of the slot (the rest of the slot up
 * to the next 16-byte boundary is written with zeros, later bytes are untouched);
 * other rows hold their raw bytes. d_row_bitmask (ceil(n_rows/32) words) is fully
 * rewritten, bits past n_rows set to 0. d_row_bits (nullable, n_rows words)
 * receives each row's size-formula bit count. rows and slots must not overlap. */
int ibp_compress(const void *rows, int64_t n_rows, int64_t row_elems, int dtype,
                 uint32_t block_elems, const ibp_meta *d_meta, void *slots, int64_t slot_bytes,
                 uint32_t *d_row_bitmask, uint32_t *d_row_bits, int32_t *d_status,
                 ibp_stream_t s);

/* Decompress-gather ("Core algorithm", decompression; "System integration").
 * out[i] (row_elems words, device memory, rows packed back to back) receives the
 * original row d_idx[i] for i < n_idx; indices may repeat. Only the used prefix of
 * each slot is read. n_idx == 0 is a no-op. A row whose index is outside
 * [0, n_rows) or whose participation bits describe a stream that would not have
 * been stored compressed is skipped (out[i] untouched) and IBP_ERR_INDEX or
 * IBP_ERR_CORRUPT is recorded in *d_status. */
int ibp_decompress_gather(const void *slots, int64_t slot_bytes, int64_t n_rows,
                          int64_t row_elems, int dtype, uint32_t block_elems,
                          const uint32_t *d_row_bitmask, const ibp_meta *d_meta,
                          const int64_t *d_idx, int64_t n_idx, void *out, int32_t *d_status,
                          ibp_stream_t s);

/* Packed store ("System integration": compressing a GPU cache's rows raises its
 * effective capacity; the paper has no layout for it, so this one is the
 * library's). A slotted store keeps every row in a raw-size slot (a row can be
 * rewritten in place); a packed store lays rows end to end and is read only:
 *   entry i = the used prefix of slot d_sel[i] (d_sel null: row i) -- the
 *     4*ceil(bits/32) stream bytes of a compressed row, or the raw row -- rounded up
 *     to a multiple of 16 bytes, copied from the slot (stream padding included);
 *   d_offsets[i] = byte offset of entry i; d_offsets[n_sel] = total bytes
 *     (n_sel + 1 uint64 entries, device memory).
 * Entry i of the packed store is row i: its bitmask bit and bit count are the
 * source row's. Build it in three calls: ibp_pack_offsets, read d_offsets[n_sel]
 * to size the buffer, ibp_pack. */

/* Device scratch ibp_pack_offsets needs for n_sel entries (8 bytes per 4096). */
int ibp_pack_scratch_bytes(int64_t n_sel, size_t *bytes);

/* Entry offsets of a packed store of rows d_sel[0..n_sel) of a slotted store
 * described by d_row_bitmask and d_row_bits (both as written by ibp_compress;
 * row_bits is required here). A selection outside [0, n_rows) gets a 0-byte entry
 * and IBP_ERR_INDEX in *d_status. Asynchronous on s. */
int ibp_pack_offsets(const uint32_t *d_row_bitmask, const uint32_t *d_row_bits, int64_t n_rows,
                     int64_t row_elems, int dtype, const int64_t *d_sel, int64_t n_sel,
                     uint64_t *d_offsets, void *d_scratch, int32_t *d_status, ibp_stream_t s);

/* Copy the entries into packed (device or registered host memory, packed_bytes
 * long, 16-byte aligned) and write the packed store's bitmask d_pack_bitmask
 * (ceil(n_sel/32) words, fully rewritten) and, when non-null, d_pack_row_bits
 * (n_sel words). An entry whose offsets disagree with its row's size, are not
 * 16-byte aligned or leave the buffer is skipped with IBP_ERR_CORRUPT in
 * *d_status; a bad selection with IBP_ERR_INDEX. slots and packed must not
 * overlap. */
int ibp_pack(const void *slots, int64_t slot_bytes, int64_t n_rows, int64_t row_elems, int dtype,
             const uint32_t *d_row_bitmask, const uint32_t *d_row_bits, const int64_t *d_sel,
             int64_t n_sel, const uint64_t *d_offsets, void *packed, uint64_t packed_bytes,
             uint32_t *d_pack_bitmask, uint32_t *d_pack_row_bits, int32_t *d_status,
             ibp_stream_t s);

/* ibp_decompress_gather on a packed store of n_rows entries: row r is read from
 * packed + d_offsets[r], d_offsets[r+1] - d_offsets[r] bytes of it. Rows of at most
 * 32 blocks are staged whole (exactly their entry) with no header round trip. An
 * entry whose offsets are unaligned, decreasing or past packed_bytes, or too short
 * for the row its header describes, is skipped with IBP_ERR_CORRUPT. */
int ibp_decompress_gather_packed(const void *packed, uint64_t packed_bytes,
                                 const uint64_t *d_offsets, int64_t n_rows, int64_t row_elems,
                                 int dtype, uint32_t block_elems, const uint32_t *d_row_bitmask,
                                 const ibp_meta *d_meta, const int64_t *d_idx, int64_t n_idx,
                                 void *out, int32_t *d_status, ibp_stream_t s);

/* De-duplicated decompress-gather ("Core algorithm", decompression; "System
 * integration", rows in host memory moved over the host link). Same arguments and
 * result as ibp_decompress_gather: out[i] (n_idx x row_elems words, device memory)
 * is row d_idx[i]; an index outside [0, n_rows) records IBP_ERR_INDEX in *d_status
 * and leaves its output row untouched. Each distinct row of d_idx is read from its
 * slot and decoded once, straight into the output row of one position that names it
 * (the first to claim it), then copied from there to every other position that names
 * it: for skewed index lists a row crosses the host link once instead of once per
 * request. d_scratch: device memory of scratch_bytes >= the size
 * ibp_gather_dedup_scratch_bytes reports (12 bytes per index plus a hash table of at
 * least 16 bytes per index, all rounded up), 16-byte aligned, overwritten;
 * scratch_bytes too small: IBP_ERR_ARG. n_idx up to 2^24 - 1 and n_rows below 2^40,
 * else IBP_ERR_UNSUPPORTED. Asynchronous on s: three launches (clear, a gather that
 * claims each row as it goes, copy) for rows of at most 32 blocks and 4 KiB, four (a
 * hash pass before the gather) for longer rows; allocates nothing. */
int ibp_gather_dedup_scratch_bytes(int64_t n_idx, int64_t row_elems, int dtype,
                                   uint32_t block_elems, size_t *bytes);
int ibp_decompress_gather_dedup(const void *slots, int64_t slot_bytes, int64_t n_rows,
                                int64_t row_elems, int dtype, uint32_t block_elems,
                                const uint32_t *d_row_bitmask, const ibp_meta *d_meta,
                                const int64_t *d_idx, int64_t n_idx, void *out, void *d_scratch,
                                size_t scratch_bytes, int32_t *d_status, ibp_stream_t s);

/* ibp_decompress_gather given also the per-row bit counts ibp_compress wrote
 * (d_row_bits, n_rows words, device memory). A row's stored length is then known
 * from device memory before its slot is read, so exactly its used prefix (rounded
 * up to 16 bytes) is staged, with no round trip through the slot's header: for
 * slots in host memory only the stored bytes cross the link. A bit count that
 * disagrees with the row's header is reported as IBP_ERR_CORRUPT. */
int ibp_decompress_gather_sized(const void *slots, int64_t slot_bytes, int64_t n_rows,
                                int64_t row_elems, int dtype, uint32_t block_elems,
                                const uint32_t *d_row_bitmask, const uint32_t *d_row_bits,
                                const ibp_meta *d_meta, const int64_t *d_idx, int64_t n_idx,
                                void *out, int32_t *d_status, ibp_stream_t s);

/* One gather of a batch: a store (slots, slot_bytes, n_rows, its bitmask and
 * metadata) and the indices to read from it into out, as in ibp_decompress_gather. */
typedef struct {
  const void *slots;              /* device or registered host memory, 16-byte aligned */
  int64_t slot_bytes;
  int64_t n_rows;
  const uint32_t *d_row_bitmask;  /* device */
  const ibp_meta *d_meta;         /* device */
  const int64_t *d_idx;           /* device */
  int64_t n_idx;
  void *out;                      /* device, n_idx x row_elems words, 16-byte aligned */
} ibp_gather_job;

/* Several decompress-gathers with one row geometry (row_elems, dtype, block_elems)
 * in one launch per 64 jobs: e.g. one lookup batch per embedding table of a model.
 * jobs: host array of n_jobs descriptions (read during the call; the structs need
 * not outlive it). Each job gets CTAs in proportion to its indices, so the fixed
 * cost of a launch is paid once for the batch. Per-job checks, results and device
 * errors are those of ibp_decompress_gather (*d_status is shared by all jobs). */
int ibp_decompress_gather_batched(const ibp_gather_job *jobs, int n_jobs, int64_t row_elems,
                                  int dtype, uint32_t block_elems, int32_t *d_status,
                                  ibp_stream_t s);

/* Decompress a contiguous range of rows in order: out[i] = row row_begin + i for
 * i < n_out (row_begin + n_out <= n_rows). The same as ibp_decompress_gather with
 * d_idx = row_begin, row_begin + 1, ..., without an index array: for streaming
 * whole tensors (a layer's weights, a sequence's K/V rows) out of a store. */
int ibp_decompress_range(const void *slots, int64_t slot_bytes, int64_t n_rows, int64_t row_elems,
                         int dtype, uint32_t block_elems, const uint32_t *d_row_bitmask,
                         const ibp_meta *d_meta, int64_t row_begin, int64_t n_out, void *out,
                         int32_t *d_status, ibp_stream_t s);

/* Per-position metadata (a variant of preprocessing: the "kilobyte-scale" metadata
 * reading of "Core algorithm"; the paper fixes no layout, this one is the
 * library's). Element position e of a row (0 <= e < row_elems) has its own
 * mask/bitval pair, d_pmask[e] / d_pbitval[e] (w-bit values in uint32 words,
 * device memory, row_elems entries each): the preprocessing rule of ibp_build_meta
 * applied to the sample made of element e of every row. A block matches when each
 * of its elements e satisfies (x & pmask[e]) == pbitval[e]; a matching element is
 * stored as a field of w - popcount(pmask[e]) bits (its non-invariant bits,
 * ascending). Participation bits, bit order, shorter last blocks and the store rule
 * are those of the shared-mask format. Rows of at most 16 KiB (else
 * IBP_ERR_UNSUPPORTED); the argument checks of the shared-mask calls apply.
 * ibp_meta_positions_scratch_bytes: device scratch of ibp_build_meta_positions (8
 * bytes per bit of a row). */
int ibp_meta_positions_scratch_bytes(int64_t row_elems, int dtype, size_t *bytes);

int ibp_build_meta_positions(const void *rows, int64_t n_rows, int64_t row_elems, int dtype,
                             double T, uint32_t block_elems, uint32_t *d_pmask,
                             uint32_t *d_pbitval, void *d_scratch, ibp_stream_t s);

/* Block-position metadata (the block-sized reading of the "kilobyte-scale" metadata
 * of "Core algorithm", preprocessing; the layout is the library's). Position q of a
 * block (0 <= q < block_elems) gets one mask/bitval pair: the preprocessing rule of
 * ibp_build_meta applied to the sample made of the element at position q of every
 * block of every row (a shorter last block adds only the positions it has, so the
 * sample of position q has n_rows * ceil((row_elems - q) / block_elems) elements).
 * The result is written row-sized, like ibp_build_meta_positions: d_pmask[e] and
 * d_pbitval[e] (row_elems entries each, device memory) hold the pair of position
 * e % block_elems, so ibp_compress_positions and ibp_decompress_gather_positions
 * take them as they are. Same arguments, limits, scratch
 * (ibp_meta_positions_scratch_bytes) and errors as ibp_build_meta_positions;
 * asynchronous on s. */
int ibp_build_meta_block_positions(const void *rows, int64_t n_rows, int64_t row_elems,
                                   int dtype, double T, uint32_t block_elems, uint32_t *d_pmask,
                                   uint32_t *d_pbitval, void *d_scratch, ibp_stream_t s);

/* ibp_compress with per-position metadata (no *d_meta; no device-detected errors). */
int ibp_compress_positions(const void *rows, int64_t n_rows, int64_t row_elems, int dtype,
                           uint32_t block_elems, const uint32_t *d_pmask,
                           const uint32_t *d_pbitval, void *slots, int64_t slot_bytes,
                           uint32_t *d_row_bitmask, uint32_t *d_row_bits, ibp_stream_t s);

/* ibp_decompress_gather with per-position metadata. Each requested row's slot is
 * staged whole (its raw-size prefix). */
int ibp_decompress_gather_positions(const void *slots, int64_t slot_bytes, int64_t n_rows,
                                    int64_t row_elems, int dtype, uint32_t block_elems,
                                    const uint32_t *d_row_bitmask, const uint32_t *d_pmask,
                                    const uint32_t *d_pbitval, const int64_t *d_idx,
                                    int64_t n_idx, void *out, int32_t *d_status,
                                    ibp_stream_t s);

/* Statistics of a store ("System integration": a fixed-size buffer per tensor of
 * which only the compressed part is used, and a GPU-resident bitmask of the
 * compressed tensors; the statistics say how much of the buffers is used).
 * Reduces the bitmask and the per-row bit counts written by ibp_compress
 * (d_row_bitmask: ceil(n_rows/32) words, d_row_bits: n_rows words, device memory;
 * both may be null when n_rows == 0) into
 *   n_rows, n_compressed (bitmask bits set), raw_bytes (n_rows * row bytes),
 *   stored_bytes (sum of 4*ceil(bits/32) over compressed rows plus the raw row
 *   bytes of the others), total_bits (sum of the per-row bit counts).
 * ibp_query writes them to *h_out (host memory of any kind) and synchronises s
 * before it returns, so it cannot be captured in a CUDA graph. Its kernel reduces
 * into a 40-byte array built into the library (the library allocates nothing);
 * calls in one process take a lock around the launch and the wait, so two calls
 * never share the array. Errors: null h_out, n_rows < 0, row_elems <= 0 or a
 * non-device bitmask/bit-count pointer: IBP_ERR_ARG; unknown dtype: IBP_ERR_DTYPE;
 * a failed launch, copy or synchronisation: IBP_ERR_CUDA (*h_out then unchanged).
 * ibp_query_async: the same reduction into *d_stats (device memory, 8-byte
 * aligned, overwritten), asynchronous on s, capturable; same argument errors. */
int ibp_query(const uint32_t *d_row_bitmask, const uint32_t *d_row_bits, int64_t n_rows,
              int64_t row_elems, int dtype, ibp_stats *h_out, ibp_stream_t s);
int ibp_query_async(const uint32_t *d_row_bitmask, const uint32_t *d_row_bits, int64_t n_rows,
                    int64_t row_elems, int dtype, ibp_stats *d_stats, ibp_stream_t s);

/* Measurement helper, not part of the codec: streams `bytes` (a multiple of 16)
 * from src (device or registered host memory) with 16-byte loads across the whole
 * GPU and writes one XOR checksum word to *d_sink, so a caller can time the plain
 * read bandwidth of the memory the codec reads zero-copy. */
int ibp_probe_read(const void *src, int64_t bytes, uint64_t *d_sink, ibp_stream_t s);

#ifdef __cplusplus
}
#endif
#endif
