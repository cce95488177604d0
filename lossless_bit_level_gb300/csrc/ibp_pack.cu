// Packed store of Invariant Bit Packing for sm_103a ("cache-compression mode").
//
// "Reducing the GPU Memory Bottleneck with Lossless Compression for ML --
// Extended", technical summary, "System integration": compressing the rows a GPU
// cache holds raises the cache's effective capacity. A slotted store keeps every
// row in a raw-size slot (so a row can be rewritten in place); a packed store
// lays the selected rows' used bytes end to end instead:
//   entry i = the used prefix of slot sel[i] (4*ceil(bits/32) bytes when the row is
//   stored compressed, the raw row otherwise) rounded up to 16 bytes;
//   offsets[i] = byte offset of entry i, offsets[n_sel] = total bytes.
// The 16-byte rounding keeps every entry aligned for 16-byte copies and costs at
// most 15 bytes per row.
//
// Offsets: a three-kernel exclusive scan of the entry sizes (tile sums, one-CTA
// scan of the tile sums, tile-local scans plus the tile's prefix), reading only
// the bitmask and the per-row bit counts. Copy: a warp per entry, 16-byte loads
// from the slot (device or registered host memory) and 16-byte stores.
#include <algorithm>

#include "ibp_device.cuh"
#include "ibp_internal.h"

namespace ibp {
namespace {

constexpr int PACK_THREADS = 256;
constexpr int PACK_ITEMS = 16;                         // entries per thread in the scan
constexpr int PACK_TILE = PACK_THREADS * PACK_ITEMS;  // entries per scan tile

struct SizeArgs {
  const uint32_t *bitmask;
  const uint32_t *row_bits;
  const int64_t *sel;  // nullable: identity
  int64_t n_rows, n_sel;
  int64_t raw_bytes;
  int32_t *status;
};

// Bytes of entry i of the packed store (0 for a selection outside the store).
__device__ __forceinline__ uint64_t entry_bytes(const SizeArgs &a, int64_t i) {
  const int64_t r = a.sel ? a.sel[i] : i;
  if (r < 0 || r >= a.n_rows) {
    report(a.status, IBP_ERR_INDEX);
    return 0;
  }
  const bool compressed = (a.bitmask[r >> 5] >> (r & 31)) & 1u;
  const uint64_t used =
      compressed ? 4ull * (((uint64_t)a.row_bits[r] + 31) >> 5) : (uint64_t)a.raw_bytes;
  return (used + 15) & ~15ull;
}

__device__ __forceinline__ uint64_t warp_inclusive_sum(uint64_t v) {
  const int lane = threadIdx.x & 31;
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t t = __shfl_up_sync(FULL, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Exclusive scan of one value per thread across the CTA; *total gets the sum.
__device__ __forceinline__ uint64_t cta_exclusive_sum(uint64_t v, uint64_t *warp_sums,
                                                      uint64_t *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint64_t inc = warp_inclusive_sum(v);
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const uint64_t s = lane < PACK_THREADS / 32 ? warp_sums[lane] : 0;
    const uint64_t si = warp_inclusive_sum(s);
    if (lane < PACK_THREADS / 32) warp_sums[lane] = si - s;
    if (lane == PACK_THREADS / 32 - 1) warp_sums[PACK_THREADS / 32] = si;
  }
  __syncthreads();
  const uint64_t out = warp_sums[warp] + inc - v;
  *total = warp_sums[PACK_THREADS / 32];
  __syncthreads();
  return out;
}

__global__ void __launch_bounds__(PACK_THREADS) pack_tile_sums_kernel(SizeArgs a,
                                                                      uint64_t *tile_sums) {
  __shared__ uint64_t warp_sums[PACK_THREADS / 32 + 1];
  const int64_t base = (int64_t)blockIdx.x * PACK_TILE;
  uint64_t s = 0;
  for (int k = 0; k < PACK_ITEMS; ++k) {
    const int64_t i = base + (int64_t)k * PACK_THREADS + threadIdx.x;
    if (i < a.n_sel) s += entry_bytes(a, i);
  }
  uint64_t total;
  cta_exclusive_sum(s, warp_sums, &total);
  if (threadIdx.x == 0) tile_sums[blockIdx.x] = total;
}

// One CTA: exclusive scan of the tile sums in place; offsets[n_sel] = the total.
__global__ void __launch_bounds__(PACK_THREADS) pack_scan_tiles_kernel(uint64_t *tile_sums,
                                                                       int64_t n_tiles,
                                                                       uint64_t *offsets,
                                                                       int64_t n_sel) {
  __shared__ uint64_t warp_sums[PACK_THREADS / 32 + 1];
  uint64_t carry = 0;
  for (int64_t b = 0; b < n_tiles; b += PACK_THREADS) {
    const int64_t t = b + threadIdx.x;
    const uint64_t v = t < n_tiles ? tile_sums[t] : 0;
    uint64_t total;
    const uint64_t ex = cta_exclusive_sum(v, warp_sums, &total);
    if (t < n_tiles) tile_sums[t] = carry + ex;
    carry += total;
  }
  if (threadIdx.x == 0) offsets[n_sel] = carry;
}

__global__ void __launch_bounds__(PACK_THREADS) pack_offsets_kernel(SizeArgs a,
                                                                    const uint64_t *tile_sums,
                                                                    uint64_t *offsets) {
  __shared__ uint64_t warp_sums[PACK_THREADS / 32 + 1];
  // thread t owns entries base + t*PACK_ITEMS .. + PACK_ITEMS (contiguous, so the
  // CTA scan of per-thread sums orders them)
  const int64_t first = (int64_t)blockIdx.x * PACK_TILE + (int64_t)threadIdx.x * PACK_ITEMS;
  uint64_t sz[PACK_ITEMS];
  uint64_t s = 0;
#pragma unroll
  for (int k = 0; k < PACK_ITEMS; ++k) {
    const int64_t i = first + k;
    sz[k] = i < a.n_sel ? entry_bytes(a, i) : 0;
    s += sz[k];
  }
  uint64_t total;
  uint64_t at = tile_sums[blockIdx.x] + cta_exclusive_sum(s, warp_sums, &total);
#pragma unroll
  for (int k = 0; k < PACK_ITEMS; ++k) {
    const int64_t i = first + k;
    if (i < a.n_sel) offsets[i] = at;
    at += sz[k];
  }
}

struct CopyArgs {
  const uint8_t *slots;
  int64_t slot_bytes;
  const uint32_t *bitmask;
  const uint32_t *row_bits;
  const int64_t *sel;
  int64_t n_rows, n_sel;
  int64_t raw_bytes;
  const uint64_t *offsets;
  uint8_t *packed;
  uint64_t packed_bytes;
  uint32_t *pack_bitmask;
  uint32_t *pack_row_bits;
  int32_t *status;
};

__global__ void __launch_bounds__(PACK_THREADS) pack_copy_kernel(CopyArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (PACK_THREADS / 32);
  for (int64_t i = (int64_t)blockIdx.x * (PACK_THREADS / 32) + (threadIdx.x >> 5); i < a.n_sel;
       i += warps) {
    const int64_t r = a.sel ? a.sel[i] : i;
    if (r < 0 || r >= a.n_rows) {
      if (lane == 0) report(a.status, IBP_ERR_INDEX);
      continue;
    }
    const bool compressed = (a.bitmask[r >> 5] >> (r & 31)) & 1u;
    const uint32_t bits = a.row_bits[r];
    const uint64_t used = compressed ? 4ull * (((uint64_t)bits + 31) >> 5) : (uint64_t)a.raw_bytes;
    const uint64_t len = (used + 15) & ~15ull;
    const uint64_t o0 = a.offsets[i], o1 = a.offsets[i + 1];
    // the entry must be where the offsets say, whole, aligned and inside the buffer
    if (o1 < o0 || o1 - o0 != len || (o0 & 15) || o1 > a.packed_bytes ||
        len > (uint64_t)a.slot_bytes) {
      if (lane == 0) report(a.status, IBP_ERR_CORRUPT);
      continue;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(a.slots + r * a.slot_bytes);
    uint4 *dst = reinterpret_cast<uint4 *>(a.packed + o0);
    const uint32_t nvec = (uint32_t)(len >> 4);
    for (uint32_t v = lane; v < nvec; v += 32) dst[v] = src[v];
    if (lane == 0) {
      if (compressed) atomicOr(a.pack_bitmask + (i >> 5), 1u << (i & 31));
      if (a.pack_row_bits) a.pack_row_bits[i] = bits;
    }
  }
}

}  // namespace

size_t pack_scratch_bytes(int64_t n_sel) {
  const int64_t tiles = std::max<int64_t>(1, (n_sel + PACK_TILE - 1) / PACK_TILE);
  return (size_t)tiles * sizeof(uint64_t);
}

int launch_pack_offsets(const uint32_t *d_bitmask, const uint32_t *d_row_bits, int64_t n_rows,
                        int64_t raw_bytes, const int64_t *d_sel, int64_t n_sel,
                        uint64_t *d_offsets, void *d_scratch, int32_t *d_status,
                        cudaStream_t s) {
  SizeArgs a;
  a.bitmask = d_bitmask;
  a.row_bits = d_row_bits;
  a.sel = d_sel;
  a.n_rows = n_rows;
  a.n_sel = n_sel;
  a.raw_bytes = raw_bytes;
  a.status = d_status;
  uint64_t *tile_sums = static_cast<uint64_t *>(d_scratch);
  const int64_t tiles = (n_sel + PACK_TILE - 1) / PACK_TILE;
  if (tiles > 0) {
    pack_tile_sums_kernel<<<(unsigned)tiles, PACK_THREADS, 0, s>>>(a, tile_sums);
    if (cudaGetLastError() != cudaSuccess) return IBP_ERR_CUDA;
  }
  pack_scan_tiles_kernel<<<1, PACK_THREADS, 0, s>>>(tile_sums, tiles, d_offsets, n_sel);
  if (cudaGetLastError() != cudaSuccess) return IBP_ERR_CUDA;
  if (tiles > 0) {
    pack_offsets_kernel<<<(unsigned)tiles, PACK_THREADS, 0, s>>>(a, tile_sums, d_offsets);
    if (cudaGetLastError() != cudaSuccess) return IBP_ERR_CUDA;
  }
  return IBP_OK;
}

int launch_pack(const void *slots, int64_t slot_bytes, int64_t n_rows, int64_t raw_bytes,
                const uint32_t *d_bitmask, const uint32_t *d_row_bits, const int64_t *d_sel,
                int64_t n_sel, const uint64_t *d_offsets, void *packed, uint64_t packed_bytes,
                uint32_t *d_pack_bitmask, uint32_t *d_pack_row_bits, int32_t *d_status,
                cudaStream_t s) {
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  if (n_sel == 0) return IBP_OK;
  if (cudaMemsetAsync(d_pack_bitmask, 0, (size_t)((n_sel + 31) / 32) * 4, s) != cudaSuccess)
    return IBP_ERR_CUDA;
  CopyArgs a;
  a.slots = static_cast<const uint8_t *>(slots);
  a.slot_bytes = slot_bytes;
  a.bitmask = d_bitmask;
  a.row_bits = d_row_bits;
  a.sel = d_sel;
  a.n_rows = n_rows;
  a.n_sel = n_sel;
  a.raw_bytes = raw_bytes;
  a.offsets = d_offsets;
  a.packed = static_cast<uint8_t *>(packed);
  a.packed_bytes = packed_bytes;
  a.pack_bitmask = d_pack_bitmask;
  a.pack_row_bits = d_pack_row_bits;
  a.status = d_status;
  const int64_t want = (n_sel + PACK_THREADS / 32 - 1) / (PACK_THREADS / 32);
  const int grid = (int)std::min<int64_t>(want, (int64_t)dev.sm_count * 8);
  pack_copy_kernel<<<grid, PACK_THREADS, 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

}  // namespace ibp
