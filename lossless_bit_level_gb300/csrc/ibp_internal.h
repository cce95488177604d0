// Internal declarations shared by the codec's CUDA translation units (host side).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ibp.h"

namespace ibp {

// Row geometry, computed on the host from (row_elems, dtype, block_elems).
// Kernels work on 32-bit "lane words": one FP32 element or two 16-bit elements.
struct RowGeom {
  int w;             // element width in bits (8, 16 or 32)
  int epw;           // elements per lane word (32 / w)
  int B;             // block size in elements
  int lwb;           // lane words per block (B * w / 32): 8, 16, 32 or 64
  int lwt;           // lane words of the last block (lwb, or fewer for a shorter tail)
  int nb;            // blocks per row (ceil(row_elems / B))
  int raw_words;     // lane words per row
  int64_t row_elems; // elements per row
  int64_t raw_bytes; // bytes per raw row
};

inline int width_of(int dtype) {
  return dtype == IBP_FP32 ? 32 : (dtype == IBP_W8 ? 8 : 16);
}

// Device properties the launchers size their grids with (cached per device).
struct DeviceInfo {
  int device;
  int sm_count;
  int max_smem_optin;
};
int device_info(DeviceInfo *out);

int launch_build_meta(const void *rows, int64_t n_words, int dtype, double T, uint32_t block_elems,
                      int64_t n_elems, ibp_meta *d_meta, void *d_scratch, cudaStream_t s);
// The positional population count of the preprocessing stage: clears the 32
// 64-bit counters, then adds every n_words 32-bit word into them.
int launch_meta_count(const void *rows, int64_t n_words, unsigned long long *counters,
                      cudaStream_t s);
int launch_meta_finalize(const unsigned long long *counters, int64_t n_elems, int dtype, double T,
                         uint32_t block_elems, ibp_meta *d_meta, int32_t *d_status,
                         cudaStream_t s);
int launch_build_meta_select(const void *rows, int64_t n_rows, const RowGeom &g, uint32_t dtype,
                             double T, ibp_meta *d_meta, ibp_mask_candidate *d_candidates,
                             void *d_scratch, cudaStream_t s);
size_t select_scratch_bytes();
int launch_compress(const void *rows, int64_t n_rows, const RowGeom &g, uint32_t dtype,
                    const ibp_meta *d_meta, void *slots, int64_t slot_bytes, uint32_t *d_bitmask,
                    uint32_t *d_row_bits, int32_t *d_status, cudaStream_t s);
// Rows over 2 KiB: one warp per row in one pass (the caller has checked the arguments
// and looked up the device).
int launch_compress_stream(const void *rows, int64_t n_rows, const RowGeom &g, uint32_t dtype,
                           const ibp_meta *d_meta, void *slots, int64_t slot_bytes,
                           uint32_t *d_bitmask, uint32_t *d_row_bits, int32_t *d_status,
                           const DeviceInfo &dev, cudaStream_t s);
// slots_in_device_memory selects the warp-specialised bulk-copy kernel (device
// memory) or the cp.async kernel (page-locked host memory read zero-copy).
// d_idx null: the rows row0 .. row0 + n_idx - 1 in order.
// d_row_bits non-null (slotted stores): each row's used slot prefix is known from
// device memory before the slot is read, and only that prefix is staged.
// d_offsets non-null: a packed store (entry r at slots + d_offsets[r], packed_bytes
// long in all); otherwise slot r at slots + r * slot_bytes.
// skip_negative: a negative index is a unit with nothing to do, not an error.
// pos_in_index (slotted stores only): index entries hold (output row << 40) | row.
// d_idx_count (device memory, nullable): only the first *d_idx_count index entries
// are gathered (read when the kernel starts).
// claim (nullable; slotted stores whose rows are one gather unit each): each index
// position first claims its row in claim->table (an open-addressing hash table of
// mask + 1 zeroed 64-bit slots, at least two per position): only the first position
// to claim a row decodes it, and claim->owner[i] receives the position that claimed
// row d_idx[i] (i itself for that one, -1 for a bad index).
// The gather is then launched as a programmatic dependent of the kernel before it on
// the stream (which clears the table), so that its launch overlaps that kernel.
struct ClaimTable {
  unsigned long long *table;
  uint32_t mask;
  int32_t *owner;
};
// Launch kernel<<<grid, block, smem, s>>>(args...) as a programmatic dependent of the
// previous kernel on s (the kernel must call grid_dependency_wait before it reads
// anything that kernel wrote).
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}
int gather_units_per_row(const RowGeom &g);
int launch_gather(const void *slots, int64_t slot_bytes, const uint64_t *d_offsets,
                  uint64_t packed_bytes, int64_t n_rows, const RowGeom &g, uint32_t dtype,
                  const uint32_t *d_bitmask, const ibp_meta *d_meta, const int64_t *d_idx,
                  int64_t row0, int64_t n_idx, void *out, int32_t *d_status,
                  bool slots_in_device_memory, cudaStream_t s,
                  const uint32_t *d_row_bits = nullptr, bool skip_negative = false,
                  bool pos_in_index = false,
                  const unsigned long long *d_idx_count = nullptr,
                  const ClaimTable *claim = nullptr);
// De-duplicated slotted gather: every distinct row of d_idx is read and decoded once,
// into the output row of the position that claimed it, then copied to each other
// output position that asks for it (d_scratch holds the claim table and lists).
size_t dedup_scratch_bytes(int64_t n_idx, const RowGeom &g);
int64_t dedup_max_indices();  // index positions share a 64-bit word with the row
int launch_gather_dedup(const void *slots, int64_t slot_bytes, int64_t n_rows, const RowGeom &g,
                        uint32_t dtype, const uint32_t *d_bitmask, const ibp_meta *d_meta,
                        const int64_t *d_idx, int64_t n_idx, void *out, void *d_scratch,
                        int32_t *d_status, bool slots_in_device_memory, cudaStream_t s);
// Several slotted gathers with one row geometry in one launch per 64 jobs; in_device[j]:
// job j's slots are in device memory.
int launch_gather_batched(const ibp_gather_job *jobs, int n_jobs, const RowGeom &g,
                          uint32_t dtype, int32_t *d_status, const bool *in_device,
                          cudaStream_t s);
size_t pack_scratch_bytes(int64_t n_sel);
size_t pos_scratch_bytes(const RowGeom &g);
// per_block_position: one pair per position within a block, written row-sized.
int launch_build_meta_positions(const void *rows, int64_t n_rows, const RowGeom &g, double T,
                                uint32_t *d_pmask, uint32_t *d_pbitval, void *d_scratch,
                                cudaStream_t s, bool per_block_position = false);
int launch_compress_positions(const void *rows, int64_t n_rows, const RowGeom &g,
                              const uint32_t *d_pmask, const uint32_t *d_pbitval, void *slots,
                              int64_t slot_bytes, uint32_t *d_bitmask, uint32_t *d_row_bits,
                              cudaStream_t s);
int launch_gather_positions(const void *slots, int64_t slot_bytes, int64_t n_rows,
                            const RowGeom &g, const uint32_t *d_bitmask, const uint32_t *d_pmask,
                            const uint32_t *d_pbitval, const int64_t *d_idx, int64_t n_idx,
                            void *out, int32_t *d_status, cudaStream_t s);
int launch_pack_offsets(const uint32_t *d_bitmask, const uint32_t *d_row_bits, int64_t n_rows,
                        int64_t raw_bytes, const int64_t *d_sel, int64_t n_sel,
                        uint64_t *d_offsets, void *d_scratch, int32_t *d_status,
                        cudaStream_t s);
int launch_pack(const void *slots, int64_t slot_bytes, int64_t n_rows, int64_t raw_bytes,
                const uint32_t *d_bitmask, const uint32_t *d_row_bits, const int64_t *d_sel,
                int64_t n_sel, const uint64_t *d_offsets, void *packed, uint64_t packed_bytes,
                uint32_t *d_pack_bitmask, uint32_t *d_pack_row_bits, int32_t *d_status,
                cudaStream_t s);
int launch_query(const uint32_t *d_bitmask, const uint32_t *d_row_bits, int64_t n_rows,
                 int64_t raw_bytes, ibp_stats *d_stats, cudaStream_t s);
// The same reduction into a result array built into the library, copied to *h_out;
// synchronises s.
int launch_query_sync(const uint32_t *d_bitmask, const uint32_t *d_row_bits, int64_t n_rows,
                      int64_t raw_bytes, ibp_stats *h_out, cudaStream_t s);
int launch_probe_read(const void *src, int64_t bytes, uint64_t *d_sink, cudaStream_t s);
// Limit of each bounded wait inside the gather kernels launched from now on (ns of
// global time): WAIT_TIMEOUT_NS unless ibp_testing_set_wait_limit_ns set another.
uint64_t gather_wait_limit_ns();

}  // namespace ibp
