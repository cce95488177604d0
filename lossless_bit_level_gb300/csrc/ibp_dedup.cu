// De-duplicated decompress-gather for sm_103a.
//
// "Reducing the GPU Memory Bottleneck with Lossless Compression for ML --
// Extended", technical summary, "Core algorithm" (decompression of the rows an
// index list selects) and "System integration" (rows kept compressed in host memory
// and moved over the host link). The output is that of the plain gather: out[i] is
// row idx[i]. What changes is how often a row crosses the link: skewed index lists
// (Zipf-distributed lookups) name the same hot rows many times, and requests for a
// row that is already in flight miss in L2 and cross again. Here every distinct row
// is read and decoded once:
//   1. dedup_init_kernel clears the hash table and the counter and fills the compact
//      row list with -1 (one launch);
//   2. dedup_insert_kernel: an open-addressing hash table in device memory maps each
//      row to the first position that inserts it (one 64-bit compare-and-swap holds
//      row and position together, so the owner is fixed by a single atomic); the
//      owners take consecutive entries of the compact row list (one atomic per warp),
//      each entry holding the row and its owner's output position;
//   3. the slotted gather kernel decodes the compact list straight into the owners'
//      output rows; it reads the list's length from device memory when it starts and
//      stops there (the unused tail is -1 as well);
//   4. dedup_scatter_kernel copies each owner's output row to every other position
//      that asked for the same row (a warp per output row, 16-byte vectors).
// An index outside [0, n_rows) records IBP_ERR_INDEX and leaves its output row
// untouched, as in the plain gather.
#include <algorithm>

#include "ibp_device.cuh"
#include "ibp_internal.h"

namespace ibp {
namespace {

constexpr int DEDUP_THREADS = 256;
constexpr int POS_BITS = 24;  // positions below 2^24, rows below 2^40 share one word

__device__ __forceinline__ uint32_t table_slot(unsigned long long key, uint32_t mask) {
  return (uint32_t)((key * 0x9E3779B97F4A7C15ull) >> 32) & mask;  // Fibonacci hashing
}

__global__ void __launch_bounds__(DEDUP_THREADS)
    dedup_init_kernel(unsigned long long *table, uint32_t cap, unsigned long long *count,
                      int64_t *uidx, int64_t n_idx) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < (int64_t)cap || k < n_idx;
       k += stride) {
    if (k < (int64_t)cap) table[k] = 0ull;
    if (k < n_idx) uidx[k] = -1;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *count = 0ull;
}

__global__ void __launch_bounds__(DEDUP_THREADS)
    dedup_insert_kernel(const int64_t *__restrict__ idx, int64_t n_idx, int64_t n_rows,
                        unsigned long long *table, uint32_t mask, unsigned long long *count,
                        int32_t *owner, int64_t *uidx, int32_t *status) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  bool inserted = false;
  int64_t r = -1;
  if (i < n_idx) {
    r = __ldg(idx + i);
    if (r < 0 || r >= n_rows) {
      owner[i] = -1;
      report(status, IBP_ERR_INDEX);
    } else {
      const unsigned long long key = (unsigned long long)r + 1ull;  // 0 marks an empty slot
      const unsigned long long mine = (key << POS_BITS) | (unsigned long long)i;
      uint32_t h = table_slot(key, mask);
      int32_t own = -1;
      // the table has at least twice as many slots as positions, so a free slot or
      // the row's own entry is always found within mask + 1 probes
      for (uint32_t probe = 0; probe <= mask; ++probe) {
        const unsigned long long old = atomicCAS(&table[h], 0ull, mine);
        if (old == 0ull) {
          inserted = true;
          own = (int32_t)i;
          break;
        }
        if ((old >> POS_BITS) == key) {
          own = (int32_t)(old & ((1ull << POS_BITS) - 1));
          break;
        }
        h = (h + 1) & mask;
      }
      owner[i] = own;
    }
  }
  // the rows first seen in this warp take consecutive entries of the compact list:
  // the row in bits 0..39, the owner's output position in bits 40..63
  const uint32_t lanes = __ballot_sync(FULL, inserted);
  if (lanes) {
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(lanes) - 1;
    unsigned long long base = 0;
    if (lane == leader) base = atomicAdd(count, (unsigned long long)__popc(lanes));
    base = __shfl_sync(FULL, base, leader);
    if (inserted) {
      const unsigned long long k = base + (unsigned long long)__popc(lanes & low_mask(lane));
      uidx[k] = (i << 40) | r;
    }
  }
}

// Every position whose row another position owns gets a copy of the owner's output row
// (which the gather wrote); owners and bad indices are left as they are.
__global__ void __launch_bounds__(DEDUP_THREADS)
    dedup_scatter_kernel(const int32_t *__restrict__ owner, int64_t n_idx, int nvec_row,
                         uint4 *out) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (DEDUP_THREADS / 32);
  for (int64_t i = (int64_t)blockIdx.x * (DEDUP_THREADS / 32) + (threadIdx.x >> 5); i < n_idx;
       i += warps) {
    const int32_t o = __ldg(owner + i);
    if (o < 0 || o == i) continue;  // bad index, or the row's owner (written by the gather)
    const uint4 *src = out + (int64_t)o * nvec_row;
    uint4 *dst = out + i * nvec_row;
    for (int v = lane; v < nvec_row; v += 32) dst[v] = src[v];
  }
}

struct DedupLayout {
  uint32_t cap;  // hash table slots (a power of two, at least 2 * n_idx)
  size_t table, count, owner, uidx, total;  // byte offsets
};

size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

DedupLayout dedup_layout(int64_t n_idx, const RowGeom &) {
  DedupLayout L;
  uint32_t cap = 256;
  while ((int64_t)cap < 2 * n_idx) cap <<= 1;
  L.cap = cap;
  L.table = 0;
  L.count = L.table + align16((size_t)cap * 8);
  L.owner = L.count + 16;
  L.uidx = L.owner + align16((size_t)n_idx * 4);
  L.total = L.uidx + align16((size_t)n_idx * 8);
  return L;
}

}  // namespace

int64_t dedup_max_indices() { return (int64_t(1) << POS_BITS) - 1; }

size_t dedup_scratch_bytes(int64_t n_idx, const RowGeom &g) { return dedup_layout(n_idx, g).total; }

int launch_gather_dedup(const void *slots, int64_t slot_bytes, int64_t n_rows, const RowGeom &g,
                        uint32_t dtype, const uint32_t *d_bitmask, const ibp_meta *d_meta,
                        const int64_t *d_idx, int64_t n_idx, void *out, void *d_scratch,
                        int32_t *d_status, bool slots_in_device_memory, cudaStream_t s) {
  if (n_idx == 0) return IBP_OK;
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  const DedupLayout L = dedup_layout(n_idx, g);
  uint8_t *base = static_cast<uint8_t *>(d_scratch);
  auto *table = reinterpret_cast<unsigned long long *>(base + L.table);
  auto *count = reinterpret_cast<unsigned long long *>(base + L.count);
  auto *owner = reinterpret_cast<int32_t *>(base + L.owner);
  auto *uidx = reinterpret_cast<int64_t *>(base + L.uidx);
  const int init_grid = (int)std::min<int64_t>(
      (std::max<int64_t>(L.cap, n_idx) + DEDUP_THREADS - 1) / DEDUP_THREADS,
      (int64_t)dev.sm_count * 8);
  dedup_init_kernel<<<init_grid, DEDUP_THREADS, 0, s>>>(table, L.cap, count, uidx, n_idx);
  if (cudaGetLastError() != cudaSuccess) return IBP_ERR_CUDA;
  const int64_t blocks = (n_idx + DEDUP_THREADS - 1) / DEDUP_THREADS;
  dedup_insert_kernel<<<(unsigned)blocks, DEDUP_THREADS, 0, s>>>(
      d_idx, n_idx, n_rows, table, L.cap - 1, count, owner, uidx, d_status);
  if (cudaGetLastError() != cudaSuccess) return IBP_ERR_CUDA;
  if (int rc = launch_gather(slots, slot_bytes, nullptr, 0, n_rows, g, dtype, d_bitmask, d_meta,
                             uidx, 0, n_idx, out, d_status, slots_in_device_memory, s, nullptr,
                             true, true, count))
    return rc;
  const int64_t rows_per_cta = DEDUP_THREADS / 32;
  const int grid = (int)std::min<int64_t>((n_idx + rows_per_cta - 1) / rows_per_cta,
                                          (int64_t)dev.sm_count * 8);
  dedup_scatter_kernel<<<grid, DEDUP_THREADS, 0, s>>>(owner, n_idx, (int)(g.raw_bytes / 16),
                                                      static_cast<uint4 *>(out));
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

}  // namespace ibp
