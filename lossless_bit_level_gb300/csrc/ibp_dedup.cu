// De-duplicated decompress-gather for sm_103a.
//
// "Reducing the GPU Memory Bottleneck with Lossless Compression for ML --
// Extended", technical summary, "Core algorithm" (decompression of the rows an
// index list selects) and "System integration" (rows kept compressed in host memory
// and moved over the host link). The output is that of the plain gather: out[i] is
// row idx[i]. What changes is how often a row crosses the link: skewed index lists
// (Zipf-distributed lookups) name the same hot rows many times, and requests for a
// row that is already in flight miss in L2 and cross again. Here every distinct row
// is read and decoded once, and the other positions that ask for it get a copy:
//   1. dedup_init_kernel clears an open-addressing hash table (at least two 64-bit
//      slots per position) and a counter (one launch). A slot maps a row to the first
//      position that claims it, row and position in one word, so the owner is fixed
//      by a single compare-and-swap.
//   2. Rows that are one gather unit (up to 32 blocks and 4 KiB): the slotted gather
//      runs over the index list as it is, and before planning a position it claims
//      the position's row in the table; only owners stage and decode, each into its
//      own output row, and every position records its owner.
//      Longer rows (several units each, planned independently): dedup_insert_kernel
//      claims first. Each CTA takes 1024 consecutive positions and folds repeats among
//      them in a shared-memory table, so a row that is hot across the whole list (a
//      Zipf head) costs one global atomic per CTA, not one per position; the CTA's
//      owners take consecutive entries of a compact row list (one atomic per CTA),
//      each entry holding the row and its owner's output position, and the slotted
//      gather then decodes that list straight into the owners' output rows (it reads
//      the list's length from device memory when it starts and stops there).
//   3. dedup_scatter_kernel copies each owner's output row to every other position
//      that asked for the same row (a warp per 32 consecutive positions, up to four
//      rows' 16-byte vectors in flight per lane).
// An index outside [0, n_rows) records IBP_ERR_INDEX and leaves its output row
// untouched, as in the plain gather.
#include <algorithm>

#include "ibp_device.cuh"
#include "ibp_internal.h"

namespace ibp {
namespace {

constexpr int DEDUP_THREADS = 256;
constexpr int POS_BITS = 24;  // positions below 2^24, rows below 2^40 share one word
constexpr int INS_THREADS = 1024;
constexpr int INS_PER_THREAD = 1;
constexpr int INS_CHUNK = INS_THREADS * INS_PER_THREAD;  // positions per CTA
constexpr int LOCAL_SLOTS = 2 * INS_CHUNK;                 // shared table, a power of two
constexpr int SCATTER_GROUP = 32;
constexpr int SCATTER_BATCH = 4;

__device__ __forceinline__ uint32_t table_slot(unsigned long long key, uint32_t mask) {
  return (uint32_t)((key * 0x9E3779B97F4A7C15ull) >> 32) & mask;  // Fibonacci hashing
}

__global__ void __launch_bounds__(DEDUP_THREADS)
    dedup_init_kernel(unsigned long long *table, uint32_t cap, unsigned long long *count) {
  grid_launch_dependents();  // the gather may start launching; it waits for this kernel
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < (int64_t)cap; k += stride)
    table[k] = 0ull;
  if (blockIdx.x == 0 && threadIdx.x == 0) *count = 0ull;
}

// Insert `key` (row + 1) for position i; returns the row's owner and whether i is it.
// The table has at least twice as many slots as positions, so a free slot or the
// row's own entry is always found within mask + 1 probes (the first probe's result
// comes in as `old`).
__device__ __forceinline__ int32_t global_insert(unsigned long long *table, uint32_t mask,
                                                 unsigned long long key, int64_t i, uint32_t h,
                                                 unsigned long long old, bool *inserted) {
  const unsigned long long mine = (key << POS_BITS) | (unsigned long long)i;
  for (uint32_t probe = 0; probe <= mask; ++probe) {
    if (old == 0ull) {
      *inserted = true;
      return (int32_t)i;
    }
    if ((old >> POS_BITS) == key) return (int32_t)(old & ((1ull << POS_BITS) - 1));
    h = (h + 1) & mask;
    old = atomicCAS(&table[h], 0ull, mine);
  }
  return -1;
}

__global__ void __launch_bounds__(INS_THREADS)
    dedup_insert_kernel(const int64_t *__restrict__ idx, int64_t n_idx, int64_t n_rows,
                        unsigned long long *table, uint32_t mask, unsigned long long *count,
                        int32_t *owner, int64_t *uidx, int32_t *status) {
  constexpr int WARPS = INS_THREADS / 32;
  __shared__ unsigned long long lkey[LOCAL_SLOTS];  // row + 1 (0: empty)
  __shared__ int32_t lown[LOCAL_SLOTS];             // the row's owner in the whole list
  __shared__ uint32_t wbase[WARPS];                 // compact-list entries before each warp's
  __shared__ unsigned long long cbase;              // the CTA's first compact-list entry
  for (int k = threadIdx.x; k < LOCAL_SLOTS; k += INS_THREADS) lkey[k] = 0ull;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t base = (int64_t)blockIdx.x * INS_CHUNK + threadIdx.x;
  int64_t r[INS_PER_THREAD];
#pragma unroll
  for (int j = 0; j < INS_PER_THREAD; ++j) {
    const int64_t i = base + j * INS_THREADS;
    r[j] = i < n_idx ? __ldg(idx + i) : 0;
  }
  __syncthreads();
  int lslot[INS_PER_THREAD];  // shared-table slot of each of this thread's positions
  bool lead[INS_PER_THREAD];  // first of its row within the CTA
  unsigned long long key[INS_PER_THREAD];
#pragma unroll
  for (int j = 0; j < INS_PER_THREAD; ++j) {
    const int64_t i = base + j * INS_THREADS;
    lslot[j] = -1;
    lead[j] = false;
    key[j] = 0ull;
    if (i >= n_idx) continue;
    if (r[j] < 0 || r[j] >= n_rows) {
      owner[i] = -1;
      report(status, IBP_ERR_INDEX);
      continue;
    }
    key[j] = (unsigned long long)r[j] + 1ull;
    uint32_t h = table_slot(key[j], LOCAL_SLOTS - 1);
    for (int probe = 0; probe < LOCAL_SLOTS; ++probe) {  // 2 slots per position: found
      const unsigned long long old = atomicCAS(&lkey[h], 0ull, key[j]);
      if (old == 0ull || old == key[j]) {
        lead[j] = old == 0ull;
        lslot[j] = (int)h;
        break;
      }
      h = (h + 1) & (LOCAL_SLOTS - 1);
    }
  }
  __syncthreads();
  // the CTA's distinct rows go into the global table, first probes issued together
  uint32_t h[INS_PER_THREAD];
  unsigned long long old[INS_PER_THREAD];
#pragma unroll
  for (int j = 0; j < INS_PER_THREAD; ++j) {
    h[j] = table_slot(key[j], mask);
    const unsigned long long mine = (key[j] << POS_BITS) | (unsigned long long)(base + j * INS_THREADS);
    old[j] = lead[j] ? atomicCAS(&table[h[j]], 0ull, mine) : 0ull;
  }
  bool inserted[INS_PER_THREAD];
  uint32_t mine_n = 0;
#pragma unroll
  for (int j = 0; j < INS_PER_THREAD; ++j) {
    inserted[j] = false;
    if (lead[j])
      lown[lslot[j]] = global_insert(table, mask, key[j], base + j * INS_THREADS, h[j], old[j],
                                     &inserted[j]);
    mine_n += inserted[j] ? 1u : 0u;
  }
  // the rows this CTA inserted first take consecutive entries of the compact list (one
  // atomic per CTA): the row in bits 0..39, the owner's output position in bits 40..63
  uint32_t incl = mine_n;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t y = __shfl_up_sync(FULL, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) wbase[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t t = lane < WARPS ? wbase[lane] : 0u;
    uint32_t x = t;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t y = __shfl_up_sync(FULL, x, d);
      if (lane >= d) x += y;
    }
    if (lane < WARPS) wbase[lane] = x - t;
    if (lane == 31) cbase = x ? atomicAdd(count, (unsigned long long)x) : 0ull;
  }
  __syncthreads();
  unsigned long long k = cbase + wbase[warp] + (incl - mine_n);
#pragma unroll
  for (int j = 0; j < INS_PER_THREAD; ++j)
    if (inserted[j]) uidx[k++] = ((base + j * INS_THREADS) << 40) | r[j];
#pragma unroll
  for (int j = 0; j < INS_PER_THREAD; ++j)
    if (lslot[j] >= 0) owner[base + j * INS_THREADS] = lown[lslot[j]];
}

// Every position whose row another position owns gets a copy of the owner's output row
// (which the gather wrote; an owner is never itself a copy target); owners and bad
// indices are left as they are. A warp takes 32 consecutive positions and copies the
// rows of up to four of them at a time.
__global__ void __launch_bounds__(DEDUP_THREADS)
    dedup_scatter_kernel(const int32_t *__restrict__ owner, int64_t n_idx, int nvec_row,
                         uint4 *out) {
  constexpr int GP = SCATTER_GROUP;  // positions a warp takes at a time
  constexpr int NB = SCATTER_BATCH;  // rows in flight per lane
  grid_dependency_wait();  // the gather before it wrote the owners' rows
  const int lane = threadIdx.x & 31;
  const int64_t groups = (n_idx + GP - 1) / GP;
  const int64_t warps = (int64_t)gridDim.x * (DEDUP_THREADS / 32);
  for (int64_t gi = (int64_t)blockIdx.x * (DEDUP_THREADS / 32) + (threadIdx.x >> 5); gi < groups;
       gi += warps) {
    const int64_t i = gi * GP + lane;
    const int32_t o = (lane < GP && i < n_idx) ? __ldg(owner + i) : -1;
    uint32_t m = __ballot_sync(FULL, o >= 0 && o != i);
    while (m) {
      int p[NB];
      int32_t src[NB];
#pragma unroll
      for (int t = 0; t < NB; ++t) {
        p[t] = m ? __ffs(m) - 1 : -1;
        m &= m - 1u;  // 0 stays 0
        src[t] = __shfl_sync(FULL, o, p[t] < 0 ? 0 : p[t]);
      }
      for (int v = lane; v < nvec_row; v += 32) {
        uint4 val[NB];
#pragma unroll
        for (int t = 0; t < NB; ++t)
          if (p[t] >= 0) val[t] = out[(int64_t)src[t] * nvec_row + v];
#pragma unroll
        for (int t = 0; t < NB; ++t)
          if (p[t] >= 0) out[(gi * GP + p[t]) * nvec_row + v] = val[t];
      }
    }
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
  const int init_grid = (int)std::min<int64_t>((L.cap + DEDUP_THREADS - 1) / DEDUP_THREADS,
                                               (int64_t)dev.sm_count * 8);
  dedup_init_kernel<<<init_grid, DEDUP_THREADS, 0, s>>>(table, L.cap, count);
  if (cudaGetLastError() != cudaSuccess) return IBP_ERR_CUDA;
  if (gather_units_per_row(g) == 1) {
    // rows of one gather unit: the gather claims each row itself (no hash pass)
    const ClaimTable claim{table, L.cap - 1, owner};
    if (int rc = launch_gather(slots, slot_bytes, nullptr, 0, n_rows, g, dtype, d_bitmask, d_meta,
                               d_idx, 0, n_idx, out, d_status, slots_in_device_memory, s,
                               nullptr, true, false, nullptr, &claim))
      return rc;
  } else {
    const int64_t blocks = (n_idx + INS_CHUNK - 1) / INS_CHUNK;
    dedup_insert_kernel<<<(unsigned)blocks, INS_THREADS, 0, s>>>(
        d_idx, n_idx, n_rows, table, L.cap - 1, count, owner, uidx, d_status);
    if (cudaGetLastError() != cudaSuccess) return IBP_ERR_CUDA;
    if (int rc = launch_gather(slots, slot_bytes, nullptr, 0, n_rows, g, dtype, d_bitmask,
                               d_meta, uidx, 0, n_idx, out, d_status, slots_in_device_memory, s,
                               nullptr, true, true, count))
      return rc;
  }
  const int64_t positions_per_cta = SCATTER_GROUP * (DEDUP_THREADS / 32);
  const int grid = (int)std::min<int64_t>((n_idx + positions_per_cta - 1) / positions_per_cta,
                                          (int64_t)dev.sm_count * 8);
  if (launch_dependent(dedup_scatter_kernel, dim3(grid), dim3(DEDUP_THREADS), 0, s,
                       static_cast<const int32_t *>(owner), n_idx, (int)(g.raw_bytes / 16),
                       static_cast<uint4 *>(out)) != cudaSuccess)
    return IBP_ERR_CUDA;
  return IBP_OK;
}

}  // namespace ibp
