// C ABI of the IBP codec: argument checks, geometry, launches (declared in include/ibp.h).
// Also holds the two small auxiliary kernels: store statistics and the read probe.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <memory>
#include <mutex>
#include <vector>

#include "ibp_device.cuh"
#include "ibp_internal.h"

namespace ibp {

namespace {

constexpr int64_t MAX_ROW_ELEMS = int64_t(1) << 20;
constexpr int BATCH_JOBS_MAX_CHECK = 256;  // job flags kept on the stack up to this many

enum class Where { device_only, device_or_host };

// Device memory, managed memory, or (when allowed) page-locked host memory that
// CUDA has mapped; anything else is rejected before a kernel could fault on it.
bool pointer_ok(const void *p, Where where, size_t align) {
  if (!p || (reinterpret_cast<uintptr_t>(p) % align) != 0) return false;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  switch (attr.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged: return true;
    case cudaMemoryTypeHost: return where == Where::device_or_host && attr.devicePointer == p;
    default: return false;
  }
}

bool in_device_memory(const void *p) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return attr.type == cudaMemoryTypeDevice;
}

bool dtype_ok(int dtype) {
  return dtype == IBP_FP32 || dtype == IBP_FP16 || dtype == IBP_BF16 || dtype == IBP_W8;
}

int make_geom(int64_t row_elems, int dtype, uint32_t block_elems, RowGeom *g) {
  if (!dtype_ok(dtype)) return IBP_ERR_DTYPE;
  if (row_elems <= 0 || block_elems == 0) return IBP_ERR_ARG;
  if (block_elems != 32 && block_elems != 64) return IBP_ERR_UNSUPPORTED;
  if (row_elems > MAX_ROW_ELEMS) return IBP_ERR_UNSUPPORTED;
  const int w = width_of(dtype);
  // a shorter last block is allowed when the row is a whole number of 16-byte
  // vectors (the kernels move rows in 16-byte pieces)
  if (row_elems % block_elems != 0 && (row_elems * w / 8) % 16 != 0) return IBP_ERR_ARG;
  g->w = w;
  g->epw = 32 / g->w;
  g->B = (int)block_elems;
  g->lwb = (int)block_elems * g->w / 32;
  g->nb = (int)((row_elems + block_elems - 1) / block_elems);
  g->lwt = (int)((row_elems - (int64_t)(g->nb - 1) * block_elems) * g->w / 32);
  g->raw_words = (int)(row_elems * g->w / 32);
  g->row_elems = row_elems;
  g->raw_bytes = row_elems * g->w / 8;
  return IBP_OK;
}

int64_t slot_bytes_of(const RowGeom &g) { return (g.raw_bytes + 15) / 16 * 16; }

__global__ void query_kernel(const uint32_t *bitmask, const uint32_t *row_bits, int64_t n_rows,
                             int64_t raw_bytes, ibp_stats *stats) {
  unsigned long long comp = 0, stored = 0, bits = 0;
  for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < n_rows;
       r += (int64_t)gridDim.x * blockDim.x) {
    const bool c = (bitmask[r >> 5] >> (r & 31)) & 1u;
    const uint32_t b = row_bits[r];
    comp += c;
    stored += c ? 4ull * ((b + 31u) >> 5) : (unsigned long long)raw_bytes;
    bits += b;
  }
  for (int o = 16; o > 0; o >>= 1) {
    comp += __shfl_xor_sync(FULL, comp, o);
    stored += __shfl_xor_sync(FULL, stored, o);
    bits += __shfl_xor_sync(FULL, bits, o);
  }
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(reinterpret_cast<unsigned long long *>(&stats->n_compressed), comp);
    atomicAdd(reinterpret_cast<unsigned long long *>(&stats->stored_bytes), stored);
    atomicAdd(reinterpret_cast<unsigned long long *>(&stats->total_bits), bits);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    stats->n_rows = n_rows;
    stats->raw_bytes = n_rows * raw_bytes;
  }
}

__global__ void probe_read_kernel(const uint4 *__restrict__ src, int64_t nvec,
                                  unsigned long long *sink) {
  uint32_t acc = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; k + 3 * stride < nvec; k += 4 * stride) {
    const uint4 a = src[k], b = src[k + stride], c = src[k + 2 * stride], d = src[k + 3 * stride];
    acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^
           d.z ^ d.w;
  }
  for (; k < nvec; k += stride) {
    const uint4 a = src[k];
    acc ^= a.x ^ a.y ^ a.z ^ a.w;
  }
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(FULL, acc, o);
  if ((threadIdx.x & 31) == 0 && acc) atomicXor(sink, (unsigned long long)acc);
}

}  // namespace

int device_info(DeviceInfo *out) {
  static DeviceInfo cache[64];
  static std::atomic<bool> have[64];  // cache[d] is complete once have[d] is set
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IBP_ERR_CUDA;
  if (dev >= 0 && dev < 64 && have[dev].load(std::memory_order_acquire)) {
    *out = cache[dev];
    return IBP_OK;
  }
  DeviceInfo d;
  d.device = dev;
  if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
          cudaSuccess)
    return IBP_ERR_CUDA;
  if (dev >= 0 && dev < 64 && !have[dev].load(std::memory_order_acquire)) {
    static std::mutex fill;
    std::lock_guard<std::mutex> lock(fill);
    if (!have[dev].load(std::memory_order_relaxed)) {
      cache[dev] = d;
      have[dev].store(true, std::memory_order_release);
    }
  }
  *out = d;
  return IBP_OK;
}

int launch_query(const uint32_t *d_bitmask, const uint32_t *d_row_bits, int64_t n_rows,
                 int64_t raw_bytes, ibp_stats *d_stats, cudaStream_t s) {
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  if (cudaMemsetAsync(d_stats, 0, sizeof(ibp_stats), s) != cudaSuccess) return IBP_ERR_CUDA;
  const int64_t want = std::max<int64_t>(1, (n_rows + 255) / 256);
  const int grid = (int)std::min<int64_t>(want, (int64_t)dev.sm_count * 4);
  query_kernel<<<grid, 256, 0, s>>>(d_bitmask, d_row_bits, n_rows, raw_bytes, d_stats);
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

// ibp_query's result lives in this array (one per device that loads the library):
// the synchronous form takes no caller device memory and the library allocates
// none. A process-wide lock is held from the clear to the end of the wait, so two
// calls never use the array at the same time. Its address is looked up on every
// call (a table lookup in the runtime), which stays right across device resets.
static __device__ __align__(16) ibp_stats g_query_result;
static std::mutex g_query_mutex;

int launch_query_sync(const uint32_t *d_bitmask, const uint32_t *d_row_bits, int64_t n_rows,
                      int64_t raw_bytes, ibp_stats *h_out, cudaStream_t s) {
  std::lock_guard<std::mutex> lock(g_query_mutex);
  void *d = nullptr;
  if (cudaGetSymbolAddress(&d, g_query_result) != cudaSuccess || !d) {
    cudaGetLastError();
    return IBP_ERR_CUDA;
  }
  ibp_stats *d_stats = static_cast<ibp_stats *>(d);
  if (int rc = launch_query(d_bitmask, d_row_bits, n_rows, raw_bytes, d_stats, s)) return rc;
  ibp_stats host;
  if (cudaMemcpyAsync(&host, d_stats, sizeof(ibp_stats), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return IBP_ERR_CUDA;
  }
  *h_out = host;
  return IBP_OK;
}

int launch_probe_read(const void *src, int64_t bytes, uint64_t *d_sink, cudaStream_t s) {
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  if (cudaMemsetAsync(d_sink, 0, sizeof(uint64_t), s) != cudaSuccess) return IBP_ERR_CUDA;
  const int64_t nvec = bytes / 16;
  if (nvec == 0) return IBP_OK;
  const int grid = (int)std::min<int64_t>((nvec + 255) / 256, (int64_t)dev.sm_count * 8);
  probe_read_kernel<<<grid, 256, 0, s>>>(static_cast<const uint4 *>(src), nvec,
                                         reinterpret_cast<unsigned long long *>(d_sink));
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

}  // namespace ibp

using namespace ibp;

extern "C" {

const char *ibp_status_string(int code) {
  switch (code) {
    case IBP_OK: return "ok";
    case IBP_ERR_ARG: return "invalid argument";
    case IBP_ERR_DTYPE: return "unknown dtype";
    case IBP_ERR_UNSUPPORTED: return "unsupported block size or row length";
    case IBP_ERR_CUDA: return "CUDA call or launch failed";
    case IBP_ERR_INDEX: return "gather index out of range";
    case IBP_ERR_CORRUPT: return "corrupt slot header";
    case IBP_ERR_META: return "metadata does not match dtype/block size";
    case IBP_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
    default: return "unknown status";
  }
}

int ibp_slot_bytes(int64_t row_elems, int dtype, int64_t *slot_bytes) {
  if (!slot_bytes) return IBP_ERR_ARG;
  if (!dtype_ok(dtype)) return IBP_ERR_DTYPE;
  if (row_elems <= 0) return IBP_ERR_ARG;
  *slot_bytes = (row_elems * width_of(dtype) / 8 + 15) / 16 * 16;
  return IBP_OK;
}

int ibp_meta_scratch_bytes(size_t *bytes) {
  if (!bytes) return IBP_ERR_ARG;
  *bytes = 32 * sizeof(unsigned long long);
  return IBP_OK;
}

int ibp_build_meta(const void *rows, int64_t n_rows, int64_t row_elems, int dtype, double T,
                   uint32_t block_elems, ibp_meta *d_meta, void *d_scratch, ibp_stream_t s) {
  RowGeom g;
  if (int rc = make_geom(row_elems, dtype, block_elems, &g)) return rc;
  if (n_rows <= 0 || !(T >= 0.0 && T <= 1.0)) return IBP_ERR_ARG;
  if (!pointer_ok(rows, Where::device_or_host, 16) || !pointer_ok(d_meta, Where::device_only, 16) ||
      !pointer_ok(d_scratch, Where::device_only, 8))
    return IBP_ERR_ARG;
  const int64_t n_elems = n_rows * row_elems;
  const int64_t n_words = n_elems * g.w / 32;
  return launch_build_meta(rows, n_words, dtype, T, block_elems, n_elems, d_meta, d_scratch,
                           reinterpret_cast<cudaStream_t>(s));
}

int ibp_meta_count(const void *rows, int64_t n_rows, int64_t row_elems, int dtype,
                   uint64_t *d_counters, ibp_stream_t s) {
  if (!dtype_ok(dtype)) return IBP_ERR_DTYPE;
  if (n_rows < 0 || row_elems <= 0 || row_elems > MAX_ROW_ELEMS) return IBP_ERR_ARG;
  const int64_t bits = n_rows * row_elems * width_of(dtype);
  if (bits % 32 != 0) return IBP_ERR_ARG;  // whole 32-bit words
  if (!pointer_ok(d_counters, Where::device_only, 8)) return IBP_ERR_ARG;
  if (n_rows > 0 && !pointer_ok(rows, Where::device_or_host, 16)) return IBP_ERR_ARG;
  return launch_meta_count(rows, bits / 32, reinterpret_cast<unsigned long long *>(d_counters),
                           reinterpret_cast<cudaStream_t>(s));
}

int ibp_meta_finalize(const uint64_t *d_counters, int64_t n_elems, int dtype, double T,
                      uint32_t block_elems, ibp_meta *d_meta, int32_t *d_status,
                      ibp_stream_t s) {
  if (!dtype_ok(dtype)) return IBP_ERR_DTYPE;
  if (n_elems <= 0 || !(T >= 0.0 && T <= 1.0)) return IBP_ERR_ARG;
  if (block_elems != 32 && block_elems != 64) return IBP_ERR_UNSUPPORTED;
  if (!pointer_ok(d_counters, Where::device_only, 8) ||
      !pointer_ok(d_meta, Where::device_only, 16) ||
      (d_status && !pointer_ok(d_status, Where::device_only, 4)))
    return IBP_ERR_ARG;
  return launch_meta_finalize(reinterpret_cast<const unsigned long long *>(d_counters), n_elems,
                              dtype, T, block_elems, d_meta, d_status,
                              reinterpret_cast<cudaStream_t>(s));
}

int ibp_meta_select_scratch_bytes(size_t *bytes) {
  if (!bytes) return IBP_ERR_ARG;
  *bytes = select_scratch_bytes();
  return IBP_OK;
}

int ibp_build_meta_select(const void *rows, int64_t n_rows, int64_t row_elems, int dtype,
                          double T, uint32_t block_elems, ibp_meta *d_meta,
                          ibp_mask_candidate *d_candidates, void *d_scratch, ibp_stream_t s) {
  RowGeom g;
  if (int rc = make_geom(row_elems, dtype, block_elems, &g)) return rc;
  if (n_rows <= 0 || !(T >= 0.0 && T <= 1.0)) return IBP_ERR_ARG;
  if (!pointer_ok(rows, Where::device_or_host, 16) || !pointer_ok(d_meta, Where::device_only, 16) ||
      !pointer_ok(d_scratch, Where::device_only, 16) ||
      (d_candidates && !pointer_ok(d_candidates, Where::device_only, 16)))
    return IBP_ERR_ARG;
  return launch_build_meta_select(rows, n_rows, g, (uint32_t)dtype, T, d_meta, d_candidates,
                                  d_scratch, reinterpret_cast<cudaStream_t>(s));
}

int ibp_compress(const void *rows, int64_t n_rows, int64_t row_elems, int dtype,
                 uint32_t block_elems, const ibp_meta *d_meta, void *slots, int64_t slot_bytes,
                 uint32_t *d_row_bitmask, uint32_t *d_row_bits, int32_t *d_status,
                 ibp_stream_t s) {
  RowGeom g;
  if (int rc = make_geom(row_elems, dtype, block_elems, &g)) return rc;
  if (n_rows < 0 || slot_bytes < slot_bytes_of(g) || slot_bytes % 16 != 0) return IBP_ERR_ARG;
  if (n_rows == 0) return IBP_OK;
  if (!pointer_ok(rows, Where::device_or_host, 16) || !pointer_ok(slots, Where::device_or_host, 16) ||
      !pointer_ok(d_meta, Where::device_only, 16) ||
      !pointer_ok(d_row_bitmask, Where::device_only, 4) ||
      (d_row_bits && !pointer_ok(d_row_bits, Where::device_only, 4)) ||
      (d_status && !pointer_ok(d_status, Where::device_only, 4)))
    return IBP_ERR_ARG;
  return launch_compress(rows, n_rows, g, (uint32_t)dtype, d_meta, slots, slot_bytes,
                         d_row_bitmask, d_row_bits, d_status, reinterpret_cast<cudaStream_t>(s));
}

int ibp_decompress_gather(const void *slots, int64_t slot_bytes, int64_t n_rows,
                          int64_t row_elems, int dtype, uint32_t block_elems,
                          const uint32_t *d_row_bitmask, const ibp_meta *d_meta,
                          const int64_t *d_idx, int64_t n_idx, void *out, int32_t *d_status,
                          ibp_stream_t s) {
  RowGeom g;
  if (int rc = make_geom(row_elems, dtype, block_elems, &g)) return rc;
  if (n_rows < 0 || n_idx < 0 || slot_bytes < slot_bytes_of(g) || slot_bytes % 16 != 0)
    return IBP_ERR_ARG;
  if (n_idx == 0) return IBP_OK;
  if (!pointer_ok(slots, Where::device_or_host, 16) ||
      !pointer_ok(d_row_bitmask, Where::device_only, 4) ||
      !pointer_ok(d_meta, Where::device_only, 16) || !pointer_ok(d_idx, Where::device_only, 8) ||
      !pointer_ok(out, Where::device_only, 16) ||
      (d_status && !pointer_ok(d_status, Where::device_only, 4)))
    return IBP_ERR_ARG;
  return launch_gather(slots, slot_bytes, nullptr, 0, n_rows, g, (uint32_t)dtype, d_row_bitmask,
                       d_meta, d_idx, 0, n_idx, out, d_status, in_device_memory(slots),
                       reinterpret_cast<cudaStream_t>(s));
}

int ibp_gather_dedup_scratch_bytes(int64_t n_idx, int64_t row_elems, int dtype,
                                   uint32_t block_elems, size_t *bytes) {
  if (!bytes) return IBP_ERR_ARG;
  RowGeom g;
  if (int rc = make_geom(row_elems, dtype, block_elems, &g)) return rc;
  if (n_idx < 0) return IBP_ERR_ARG;
  if (n_idx > dedup_max_indices()) return IBP_ERR_UNSUPPORTED;
  *bytes = dedup_scratch_bytes(n_idx, g);
  return IBP_OK;
}

int ibp_decompress_gather_dedup(const void *slots, int64_t slot_bytes, int64_t n_rows,
                                int64_t row_elems, int dtype, uint32_t block_elems,
                                const uint32_t *d_row_bitmask, const ibp_meta *d_meta,
                                const int64_t *d_idx, int64_t n_idx, void *out, void *d_scratch,
                                size_t scratch_bytes, int32_t *d_status, ibp_stream_t s) {
  RowGeom g;
  if (int rc = make_geom(row_elems, dtype, block_elems, &g)) return rc;
  if (n_rows < 0 || n_idx < 0 || slot_bytes < slot_bytes_of(g) || slot_bytes % 16 != 0)
    return IBP_ERR_ARG;
  if (n_idx > dedup_max_indices() || n_rows >= (int64_t(1) << 40)) return IBP_ERR_UNSUPPORTED;
  if (n_idx == 0) return IBP_OK;
  if (scratch_bytes < dedup_scratch_bytes(n_idx, g)) return IBP_ERR_ARG;
  if (!pointer_ok(slots, Where::device_or_host, 16) ||
      !pointer_ok(d_row_bitmask, Where::device_only, 4) ||
      !pointer_ok(d_meta, Where::device_only, 16) || !pointer_ok(d_idx, Where::device_only, 8) ||
      !pointer_ok(out, Where::device_only, 16) ||
      !pointer_ok(d_scratch, Where::device_only, 16) ||
      (d_status && !pointer_ok(d_status, Where::device_only, 4)))
    return IBP_ERR_ARG;
  return launch_gather_dedup(slots, slot_bytes, n_rows, g, (uint32_t)dtype, d_row_bitmask, d_meta,
                             d_idx, n_idx, out, d_scratch, d_status, in_device_memory(slots),
                             reinterpret_cast<cudaStream_t>(s));
}

int ibp_decompress_gather_sized(const void *slots, int64_t slot_bytes, int64_t n_rows,
                                int64_t row_elems, int dtype, uint32_t block_elems,
                                const uint32_t *d_row_bitmask, const uint32_t *d_row_bits,
                                const ibp_meta *d_meta, const int64_t *d_idx, int64_t n_idx,
                                void *out, int32_t *d_status, ibp_stream_t s) {
  RowGeom g;
  if (int rc = make_geom(row_elems, dtype, block_elems, &g)) return rc;
  if (n_rows < 0 || n_idx < 0 || slot_bytes < slot_bytes_of(g) || slot_bytes % 16 != 0)
    return IBP_ERR_ARG;
  if (n_idx == 0) return IBP_OK;
  if (!pointer_ok(slots, Where::device_or_host, 16) ||
      !pointer_ok(d_row_bitmask, Where::device_only, 4) ||
      !pointer_ok(d_row_bits, Where::device_only, 4) ||
      !pointer_ok(d_meta, Where::device_only, 16) || !pointer_ok(d_idx, Where::device_only, 8) ||
      !pointer_ok(out, Where::device_only, 16) ||
      (d_status && !pointer_ok(d_status, Where::device_only, 4)))
    return IBP_ERR_ARG;
  return launch_gather(slots, slot_bytes, nullptr, 0, n_rows, g, (uint32_t)dtype, d_row_bitmask,
                       d_meta, d_idx, 0, n_idx, out, d_status, in_device_memory(slots),
                       reinterpret_cast<cudaStream_t>(s), d_row_bits);
}

int ibp_decompress_gather_batched(const ibp_gather_job *jobs, int n_jobs, int64_t row_elems,
                                  int dtype, uint32_t block_elems, int32_t *d_status,
                                  ibp_stream_t s) {
  RowGeom g;
  if (int rc = make_geom(row_elems, dtype, block_elems, &g)) return rc;
  if (n_jobs < 0 || (n_jobs > 0 && !jobs)) return IBP_ERR_ARG;
  int64_t total_idx = 0;
  for (int j = 0; j < n_jobs; ++j) total_idx += jobs[j].n_idx > 0 ? jobs[j].n_idx : 0;
  if (total_idx == 0) {  // nothing to gather (negative counts are still refused)
    for (int j = 0; j < n_jobs; ++j)
      if (jobs[j].n_idx < 0) return IBP_ERR_ARG;
    return IBP_OK;
  }
  if (d_status && !pointer_ok(d_status, Where::device_only, 4)) return IBP_ERR_ARG;
  bool in_dev[BATCH_JOBS_MAX_CHECK];
  bool *in_device = in_dev;
  std::unique_ptr<bool[]> heap;
  if (n_jobs > BATCH_JOBS_MAX_CHECK) {
    heap.reset(new bool[(size_t)n_jobs]);
    in_device = heap.get();
  }
  for (int j = 0; j < n_jobs; ++j) {
    const ibp_gather_job &jb = jobs[j];
    if (jb.n_rows < 0 || jb.n_idx < 0 || jb.slot_bytes < slot_bytes_of(g) ||
        jb.slot_bytes % 16 != 0)
      return IBP_ERR_ARG;
    in_device[j] = false;
    if (jb.n_idx == 0) continue;
    if (!pointer_ok(jb.slots, Where::device_or_host, 16) ||
        !pointer_ok(jb.d_row_bitmask, Where::device_only, 4) ||
        !pointer_ok(jb.d_meta, Where::device_only, 16) ||
        !pointer_ok(jb.d_idx, Where::device_only, 8) || !pointer_ok(jb.out, Where::device_only, 16))
      return IBP_ERR_ARG;
    in_device[j] = in_device_memory(jb.slots);
  }
  return launch_gather_batched(jobs, n_jobs, g, (uint32_t)dtype, d_status, in_device,
                               reinterpret_cast<cudaStream_t>(s));
}

int ibp_decompress_range(const void *slots, int64_t slot_bytes, int64_t n_rows, int64_t row_elems,
                         int dtype, uint32_t block_elems, const uint32_t *d_row_bitmask,
                         const ibp_meta *d_meta, int64_t row_begin, int64_t n_out, void *out,
                         int32_t *d_status, ibp_stream_t s) {
  RowGeom g;
  if (int rc = make_geom(row_elems, dtype, block_elems, &g)) return rc;
  if (n_rows < 0 || n_out < 0 || row_begin < 0 || row_begin > n_rows ||
      n_out > n_rows - row_begin || slot_bytes < slot_bytes_of(g) || slot_bytes % 16 != 0)
    return IBP_ERR_ARG;
  if (n_out == 0) return IBP_OK;
  if (!pointer_ok(slots, Where::device_or_host, 16) ||
      !pointer_ok(d_row_bitmask, Where::device_only, 4) ||
      !pointer_ok(d_meta, Where::device_only, 16) || !pointer_ok(out, Where::device_only, 16) ||
      (d_status && !pointer_ok(d_status, Where::device_only, 4)))
    return IBP_ERR_ARG;
  return launch_gather(slots, slot_bytes, nullptr, 0, n_rows, g, (uint32_t)dtype, d_row_bitmask,
                       d_meta, nullptr, row_begin, n_out, out, d_status, in_device_memory(slots),
                       reinterpret_cast<cudaStream_t>(s));
}

int ibp_pack_scratch_bytes(int64_t n_sel, size_t *bytes) {
  if (!bytes || n_sel < 0) return IBP_ERR_ARG;
  *bytes = pack_scratch_bytes(n_sel);
  return IBP_OK;
}

int ibp_pack_offsets(const uint32_t *d_row_bitmask, const uint32_t *d_row_bits, int64_t n_rows,
                     int64_t row_elems, int dtype, const int64_t *d_sel, int64_t n_sel,
                     uint64_t *d_offsets, void *d_scratch, int32_t *d_status, ibp_stream_t s) {
  if (!dtype_ok(dtype)) return IBP_ERR_DTYPE;
  if (n_rows < 0 || n_sel < 0 || row_elems <= 0 || row_elems > MAX_ROW_ELEMS) return IBP_ERR_ARG;
  if (!d_sel && n_sel > n_rows) return IBP_ERR_ARG;
  if (!pointer_ok(d_offsets, Where::device_only, 8) || !pointer_ok(d_scratch, Where::device_only, 8) ||
      (d_status && !pointer_ok(d_status, Where::device_only, 4)))
    return IBP_ERR_ARG;
  if (n_sel > 0 && (!pointer_ok(d_row_bitmask, Where::device_only, 4) ||
                    !pointer_ok(d_row_bits, Where::device_only, 4) ||
                    (d_sel && !pointer_ok(d_sel, Where::device_only, 8))))
    return IBP_ERR_ARG;
  return launch_pack_offsets(d_row_bitmask, d_row_bits, n_rows, row_elems * width_of(dtype) / 8,
                             d_sel, n_sel, d_offsets, d_scratch, d_status,
                             reinterpret_cast<cudaStream_t>(s));
}

int ibp_pack(const void *slots, int64_t slot_bytes, int64_t n_rows, int64_t row_elems, int dtype,
             const uint32_t *d_row_bitmask, const uint32_t *d_row_bits, const int64_t *d_sel,
             int64_t n_sel, const uint64_t *d_offsets, void *packed, uint64_t packed_bytes,
             uint32_t *d_pack_bitmask, uint32_t *d_pack_row_bits, int32_t *d_status,
             ibp_stream_t s) {
  if (!dtype_ok(dtype)) return IBP_ERR_DTYPE;
  if (n_rows < 0 || n_sel < 0 || row_elems <= 0 || row_elems > MAX_ROW_ELEMS) return IBP_ERR_ARG;
  const int64_t raw_bytes = row_elems * width_of(dtype) / 8;
  if (slot_bytes < (raw_bytes + 15) / 16 * 16 || slot_bytes % 16 != 0) return IBP_ERR_ARG;
  if (!d_sel && n_sel > n_rows) return IBP_ERR_ARG;
  if (n_sel == 0) return IBP_OK;
  if (!pointer_ok(slots, Where::device_or_host, 16) || !pointer_ok(packed, Where::device_or_host, 16) ||
      !pointer_ok(d_row_bitmask, Where::device_only, 4) ||
      !pointer_ok(d_row_bits, Where::device_only, 4) ||
      (d_sel && !pointer_ok(d_sel, Where::device_only, 8)) ||
      !pointer_ok(d_offsets, Where::device_only, 8) ||
      !pointer_ok(d_pack_bitmask, Where::device_only, 4) ||
      (d_pack_row_bits && !pointer_ok(d_pack_row_bits, Where::device_only, 4)) ||
      (d_status && !pointer_ok(d_status, Where::device_only, 4)))
    return IBP_ERR_ARG;
  return launch_pack(slots, slot_bytes, n_rows, raw_bytes, d_row_bitmask, d_row_bits, d_sel, n_sel,
                     d_offsets, packed, packed_bytes, d_pack_bitmask, d_pack_row_bits, d_status,
                     reinterpret_cast<cudaStream_t>(s));
}

int ibp_decompress_gather_packed(const void *packed, uint64_t packed_bytes,
                                 const uint64_t *d_offsets, int64_t n_rows, int64_t row_elems,
                                 int dtype, uint32_t block_elems, const uint32_t *d_row_bitmask,
                                 const ibp_meta *d_meta, const int64_t *d_idx, int64_t n_idx,
                                 void *out, int32_t *d_status, ibp_stream_t s) {
  RowGeom g;
  if (int rc = make_geom(row_elems, dtype, block_elems, &g)) return rc;
  if (n_rows < 0 || n_idx < 0) return IBP_ERR_ARG;
  if (n_idx == 0) return IBP_OK;
  if (!pointer_ok(packed, Where::device_or_host, 16) ||
      !pointer_ok(d_offsets, Where::device_only, 8) ||
      !pointer_ok(d_row_bitmask, Where::device_only, 4) ||
      !pointer_ok(d_meta, Where::device_only, 16) || !pointer_ok(d_idx, Where::device_only, 8) ||
      !pointer_ok(out, Where::device_only, 16) ||
      (d_status && !pointer_ok(d_status, Where::device_only, 4)))
    return IBP_ERR_ARG;
  return launch_gather(packed, 0, d_offsets, packed_bytes, n_rows, g, (uint32_t)dtype,
                       d_row_bitmask, d_meta, d_idx, 0, n_idx, out, d_status,
                       in_device_memory(packed), reinterpret_cast<cudaStream_t>(s));
}

// Per-position variant: rows of at most 16 KiB (the per-lane-word tables and two
// staged rows per warp live in shared memory).
constexpr int64_t POS_MAX_ROW_BYTES = 16384;

int ibp_meta_positions_scratch_bytes(int64_t row_elems, int dtype, size_t *bytes) {
  if (!bytes) return IBP_ERR_ARG;
  if (!dtype_ok(dtype)) return IBP_ERR_DTYPE;
  if (row_elems <= 0 || row_elems > MAX_ROW_ELEMS) return IBP_ERR_ARG;
  // one 64-bit counter per bit of a row's 32-bit lane words
  *bytes = (size_t)((row_elems * width_of(dtype) + 31) / 32) * 32 * 8;
  return IBP_OK;
}

int ibp_build_meta_positions(const void *rows, int64_t n_rows, int64_t row_elems, int dtype,
                             double T, uint32_t block_elems, uint32_t *d_pmask,
                             uint32_t *d_pbitval, void *d_scratch, ibp_stream_t s) {
  RowGeom g;
  if (int rc = make_geom(row_elems, dtype, block_elems, &g)) return rc;
  if (g.raw_bytes > POS_MAX_ROW_BYTES) return IBP_ERR_UNSUPPORTED;
  if (n_rows <= 0 || !(T >= 0.0 && T <= 1.0)) return IBP_ERR_ARG;
  if (!pointer_ok(rows, Where::device_or_host, 16) || !pointer_ok(d_pmask, Where::device_only, 4) ||
      !pointer_ok(d_pbitval, Where::device_only, 4) ||
      !pointer_ok(d_scratch, Where::device_only, 8))
    return IBP_ERR_ARG;
  return launch_build_meta_positions(rows, n_rows, g, T, d_pmask, d_pbitval, d_scratch,
                                     reinterpret_cast<cudaStream_t>(s));
}

int ibp_build_meta_block_positions(const void *rows, int64_t n_rows, int64_t row_elems,
                                   int dtype, double T, uint32_t block_elems, uint32_t *d_pmask,
                                   uint32_t *d_pbitval, void *d_scratch, ibp_stream_t s) {
  RowGeom g;
  if (int rc = make_geom(row_elems, dtype, block_elems, &g)) return rc;
  if (g.raw_bytes > POS_MAX_ROW_BYTES) return IBP_ERR_UNSUPPORTED;
  if (n_rows <= 0 || !(T >= 0.0 && T <= 1.0)) return IBP_ERR_ARG;
  if (!pointer_ok(rows, Where::device_or_host, 16) || !pointer_ok(d_pmask, Where::device_only, 4) ||
      !pointer_ok(d_pbitval, Where::device_only, 4) ||
      !pointer_ok(d_scratch, Where::device_only, 8))
    return IBP_ERR_ARG;
  return launch_build_meta_positions(rows, n_rows, g, T, d_pmask, d_pbitval, d_scratch,
                                     reinterpret_cast<cudaStream_t>(s), true);
}

int ibp_compress_positions(const void *rows, int64_t n_rows, int64_t row_elems, int dtype,
                           uint32_t block_elems, const uint32_t *d_pmask,
                           const uint32_t *d_pbitval, void *slots, int64_t slot_bytes,
                           uint32_t *d_row_bitmask, uint32_t *d_row_bits, ibp_stream_t s) {
  RowGeom g;
  if (int rc = make_geom(row_elems, dtype, block_elems, &g)) return rc;
  if (g.raw_bytes > POS_MAX_ROW_BYTES) return IBP_ERR_UNSUPPORTED;
  if (n_rows < 0 || slot_bytes < slot_bytes_of(g) || slot_bytes % 16 != 0) return IBP_ERR_ARG;
  if (n_rows == 0) return IBP_OK;
  if (!pointer_ok(rows, Where::device_or_host, 16) || !pointer_ok(slots, Where::device_or_host, 16) ||
      !pointer_ok(d_pmask, Where::device_only, 4) || !pointer_ok(d_pbitval, Where::device_only, 4) ||
      !pointer_ok(d_row_bitmask, Where::device_only, 4) ||
      (d_row_bits && !pointer_ok(d_row_bits, Where::device_only, 4)))
    return IBP_ERR_ARG;
  return launch_compress_positions(rows, n_rows, g, d_pmask, d_pbitval, slots, slot_bytes,
                                   d_row_bitmask, d_row_bits, reinterpret_cast<cudaStream_t>(s));
}

int ibp_decompress_gather_positions(const void *slots, int64_t slot_bytes, int64_t n_rows,
                                    int64_t row_elems, int dtype, uint32_t block_elems,
                                    const uint32_t *d_row_bitmask, const uint32_t *d_pmask,
                                    const uint32_t *d_pbitval, const int64_t *d_idx,
                                    int64_t n_idx, void *out, int32_t *d_status,
                                    ibp_stream_t s) {
  RowGeom g;
  if (int rc = make_geom(row_elems, dtype, block_elems, &g)) return rc;
  if (g.raw_bytes > POS_MAX_ROW_BYTES) return IBP_ERR_UNSUPPORTED;
  if (n_rows < 0 || n_idx < 0 || slot_bytes < slot_bytes_of(g) || slot_bytes % 16 != 0)
    return IBP_ERR_ARG;
  if (n_idx == 0) return IBP_OK;
  if (!pointer_ok(slots, Where::device_or_host, 16) ||
      !pointer_ok(d_row_bitmask, Where::device_only, 4) ||
      !pointer_ok(d_pmask, Where::device_only, 4) || !pointer_ok(d_pbitval, Where::device_only, 4) ||
      !pointer_ok(d_idx, Where::device_only, 8) || !pointer_ok(out, Where::device_only, 16) ||
      (d_status && !pointer_ok(d_status, Where::device_only, 4)))
    return IBP_ERR_ARG;
  return launch_gather_positions(slots, slot_bytes, n_rows, g, d_row_bitmask, d_pmask, d_pbitval,
                                 d_idx, n_idx, out, d_status, reinterpret_cast<cudaStream_t>(s));
}

static int query_args_ok(const uint32_t *d_row_bitmask, const uint32_t *d_row_bits,
                         int64_t n_rows, int64_t row_elems, int dtype) {
  if (!dtype_ok(dtype)) return IBP_ERR_DTYPE;
  if (n_rows < 0 || row_elems <= 0) return IBP_ERR_ARG;
  if (n_rows > 0 && (!pointer_ok(d_row_bitmask, Where::device_only, 4) ||
                     !pointer_ok(d_row_bits, Where::device_only, 4)))
    return IBP_ERR_ARG;
  return IBP_OK;
}

int ibp_query_async(const uint32_t *d_row_bitmask, const uint32_t *d_row_bits, int64_t n_rows,
                    int64_t row_elems, int dtype, ibp_stats *d_stats, ibp_stream_t s) {
  if (int rc = query_args_ok(d_row_bitmask, d_row_bits, n_rows, row_elems, dtype)) return rc;
  if (!pointer_ok(d_stats, Where::device_only, 8)) return IBP_ERR_ARG;
  return launch_query(d_row_bitmask, d_row_bits, n_rows, row_elems * width_of(dtype) / 8, d_stats,
                      reinterpret_cast<cudaStream_t>(s));
}

int ibp_query(const uint32_t *d_row_bitmask, const uint32_t *d_row_bits, int64_t n_rows,
              int64_t row_elems, int dtype, ibp_stats *h_out, ibp_stream_t s) {
  if (!h_out) return IBP_ERR_ARG;
  if (int rc = query_args_ok(d_row_bitmask, d_row_bits, n_rows, row_elems, dtype)) return rc;
  return launch_query_sync(d_row_bitmask, d_row_bits, n_rows, row_elems * width_of(dtype) / 8,
                           h_out, reinterpret_cast<cudaStream_t>(s));
}

int ibp_probe_read(const void *src, int64_t bytes, uint64_t *d_sink, ibp_stream_t s) {
  if (bytes < 0 || bytes % 16 != 0) return IBP_ERR_ARG;
  if (!pointer_ok(src, Where::device_or_host, 16) || !pointer_ok(d_sink, Where::device_only, 8))
    return IBP_ERR_ARG;
  return launch_probe_read(src, bytes, d_sink, reinterpret_cast<cudaStream_t>(s));
}

}  // extern "C"
