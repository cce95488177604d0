// Metadata (preprocessing) kernels of Invariant Bit Packing for sm_103a.
//
// "Reducing the GPU Memory Bottleneck with Lossless Compression for ML --
// Extended", technical summary, "Core algorithm" (preprocessing): find the bit
// positions that hold the same value in at least a fraction T of the sampled
// elements; emit a fixed-size mask and bitval kept in GPU memory.
//
// meta_count_kernel: a positional population count over the sample's 32-bit
// words. Each thread adds 8 words per step into bit-sliced carry-save counters
// (Harley-Seal: ones/twos/fours planes and a ripple counter of "eights"), so a
// word costs a handful of bitwise operations instead of 32 bit tests; the planes
// are flushed into 32 per-position totals every 255 steps, then reduced over the
// warp and added into 32 64-bit global counters. 8- and 16-bit elements are
// counted as parts of 32-bit words and folded in the finalize step.
// meta_finalize_kernel: one warp applies the threshold in IEEE double and writes
// the 16-byte ibp_meta.
#include <algorithm>
#include <atomic>

#include "ibp_device.cuh"
#include "ibp_internal.h"
#include "ibp_popcount.cuh"

namespace ibp {
namespace {

constexpr int META_THREADS = 256;

__global__ void __launch_bounds__(META_THREADS)
    meta_count_kernel(const uint4 *__restrict__ v, int64_t nvec, const uint32_t *tail, int ntail,
                      unsigned long long *counters) {
  Planes P;
#pragma unroll
  for (int j = 0; j < 32; ++j) P.tot[j] = 0;
  const int64_t npairs = (nvec + 1) / 2;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int steps = 0;
  int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  // four steps at a time: all eight 16-byte loads are issued before any is used
  for (; k + 3 * stride < npairs; k += 4 * stride) {
    uint4 a[4], b[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t kk = k + j * stride;
      a[j] = v[2 * kk];
      b[j] = (2 * kk + 1 < nvec) ? v[2 * kk + 1] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) add8(P, a[j], b[j]);
    steps += 4;
    if (steps >= 252) {
      flush_eights(P);
      steps = 0;
    }
  }
  for (; k < npairs; k += stride) {
    const uint4 a = v[2 * k];
    const uint4 b = (2 * k + 1 < nvec) ? v[2 * k + 1] : make_uint4(0, 0, 0, 0);
    add8(P, a, b);
    if (++steps == 255) {
      flush_eights(P);
      steps = 0;
    }
  }
  flush_eights(P);
#pragma unroll
  for (int j = 0; j < 32; ++j)
    P.tot[j] += ((P.ones >> j) & 1u) + 2u * ((P.twos >> j) & 1u) + 4u * ((P.fours >> j) & 1u);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    for (int i = 0; i < ntail; ++i) {
      const uint32_t x = tail[i];
#pragma unroll
      for (int j = 0; j < 32; ++j) P.tot[j] += (x >> j) & 1u;
    }
  }
  // warp reduction, then one 64-bit atomic per position per warp
  const int lane = threadIdx.x & 31;
  unsigned long long mine = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    unsigned long long s = P.tot[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(FULL, s, o);
    if (lane == j) mine = s;
  }
  if (mine) atomicAdd(&counters[lane], mine);
}

// Counters that exceed the element count cannot come from n_elems elements (e.g. one
// holder's element count passed with counters summed over several holders): the
// metadata is then written with no invariant position and an invalid dtype, so that
// compression and gathers with it report IBP_ERR_META instead of silently storing
// every row raw, and IBP_ERR_META is recorded in *status.
__global__ void meta_finalize_kernel(const unsigned long long *counters, int64_t n_elems, int w,
                                     double T, uint32_t dtype, uint32_t block_elems,
                                     ibp_meta *meta, int32_t *status) {
  const int j = threadIdx.x;  // one warp
  unsigned long long c1 = 0;  // element bit j: bits j, j + w, ... of the 32-bit words
  if (j < w)
    for (int q = j; q < 32; q += w) c1 += counters[q];
  const unsigned long long N = (unsigned long long)n_elems;
  const bool bad = __any_sync(FULL, c1 > N);
  const unsigned long long c0 = N - c1;
  const bool v = c1 > c0;  // a tie keeps 0
  const unsigned long long cv = v ? c1 : c0;
  const bool inv = j < w && (double)cv >= T * (double)N;
  const uint32_t mask = __ballot_sync(FULL, inv);
  const uint32_t bitval = __ballot_sync(FULL, inv && v);
  if (j == 0) {
    ibp_meta m;
    m.mask = bad ? 0u : mask;
    m.bitval = bad ? 0u : bitval;
    m.dtype = bad ? IBP_META_INVALID : dtype;
    m.block_elems = block_elems;
    *meta = m;
    if (bad) report(status, IBP_ERR_META);
  }
}

}  // namespace

int launch_meta_count(const void *rows, int64_t n_words, unsigned long long *counters,
                      cudaStream_t s) {
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  if (cudaMemsetAsync(counters, 0, 32 * sizeof(unsigned long long), s) != cudaSuccess)
    return IBP_ERR_CUDA;
  const int64_t nvec = n_words / 4;
  const int ntail = (int)(n_words - 4 * nvec);
  const uint32_t *tail = static_cast<const uint32_t *>(rows) + 4 * nvec;
  const int64_t npairs = (nvec + 1) / 2;
  const int64_t want = std::max<int64_t>(1, (npairs + META_THREADS - 1) / META_THREADS);
  // one wave of resident CTAs (the loop is grid-strided; a partial second wave
  // would run at a fraction of the occupancy)
  static std::atomic<int> occupancy[64];  // resident CTAs per SM, looked up once per device
  int per_sm = dev.device < 64 ? occupancy[dev.device].load(std::memory_order_relaxed) : 0;
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, meta_count_kernel, META_THREADS, 0) !=
            cudaSuccess ||
        n < 1)
      n = 1;
    per_sm = n;
    if (dev.device < 64) occupancy[dev.device].store(n, std::memory_order_relaxed);
  }
  const int grid = (int)std::min<int64_t>(want, (int64_t)dev.sm_count * per_sm);
  meta_count_kernel<<<grid, META_THREADS, 0, s>>>(static_cast<const uint4 *>(rows), nvec, tail,
                                                  ntail, counters);
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

int launch_meta_finalize(const unsigned long long *counters, int64_t n_elems, int dtype, double T,
                         uint32_t block_elems, ibp_meta *d_meta, int32_t *d_status,
                         cudaStream_t s) {
  meta_finalize_kernel<<<1, 32, 0, s>>>(counters, n_elems, width_of(dtype), T, (uint32_t)dtype,
                                        block_elems, d_meta, d_status);
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

int launch_build_meta(const void *rows, int64_t n_words, int dtype, double T, uint32_t block_elems,
                      int64_t n_elems, ibp_meta *d_meta, void *d_scratch, cudaStream_t s) {
  unsigned long long *counters = static_cast<unsigned long long *>(d_scratch);
  if (int rc = launch_meta_count(rows, n_words, counters, s)) return rc;
  return launch_meta_finalize(counters, n_elems, dtype, T, block_elems, d_meta, nullptr, s);
}

}  // namespace ibp

// ---------------------------------------------------------------------------
// Metadata build without any device allocation.
//
// Some callers cannot allocate device memory at the moment they need the
// metadata: a plug-in running inside a framework whose allocator owns all device
// memory and hands none of it out; a latency-critical loop in which a cudaMalloc
// (which may synchronise the device) must never happen; a system that forbids
// allocation once it has started. For them, the 256 bytes of bit-position
// counters live in the file-scope array below, which every GPU that loads this
// library keeps until the process exits.
//
// The counters are cleared on the stream at the start of every call, so a call
// never sees the previous call's counts, but all calls share this one array:
// two calls whose kernels overlap on the GPU (different streams, no ordering
// between them) race on it and both results are then undefined.
// ---------------------------------------------------------------------------
#include <mutex>

namespace {

constexpr int NOALLOC_COUNTER_WORDS = 32;  // one 64-bit counter per bit position of a 32-bit word
static __device__ __align__(256) unsigned long long g_noalloc_meta_counters[NOALLOC_COUNTER_WORDS];

constexpr int NOALLOC_MAX_DEVICES = 64;

// The looked-up address of the array on one device, and the CUDA context it
// belongs to. A device reset destroys the primary context; the next one loads the
// library's device code again, possibly at another address, so an address is
// reused only while the current context is the one it was found in.
struct NoallocEntry {
  void *ptr;
  unsigned long long ctx_id;
};
std::mutex g_noalloc_mutex;
NoallocEntry g_noalloc[NOALLOC_MAX_DEVICES] = {};

// Unique id of the calling thread's current CUDA context (driver entry points
// reached through the runtime, so the library needs no link-time driver
// dependency). False when there is no current context or the driver lacks the call.
bool current_context_id(unsigned long long *id) {
  typedef int (*GetCurrentFn)(void **);
  typedef int (*GetIdFn)(void *, unsigned long long *);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(f);
    cudaGetLastError();
  });
  if (!get_current || !get_id) return false;
  void *ctx = nullptr;
  if (get_current(&ctx) != 0 || !ctx) return false;
  return get_id(ctx, id) == 0;
}

// Device address of the counter array on the current device. The array's name is
// only a host-side stand-in in host code, so the address is looked up with the
// device current, once per device and context, and reused.
int noalloc_counters(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IBP_ERR_CUDA;
  unsigned long long id = 0;
  const bool have_id = current_context_id(&id);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  const bool cacheable = dev >= 0 && dev < NOALLOC_MAX_DEVICES;
  if (cacheable && have_id && g_noalloc[dev].ptr && g_noalloc[dev].ctx_id == id) {
    *out = g_noalloc[dev].ptr;
    return IBP_OK;
  }
  void *ptr = nullptr;  // (this also makes the device's primary context current)
  if (cudaGetSymbolAddress(&ptr, g_noalloc_meta_counters) != cudaSuccess || !ptr) {
    cudaGetLastError();
    return IBP_ERR_CUDA;
  }
  unsigned long long id_now = 0;
  if (cacheable) {
    // without a context id the address is not kept: every call looks it up again
    g_noalloc[dev].ptr = current_context_id(&id_now) ? ptr : nullptr;
    g_noalloc[dev].ctx_id = id_now;
  }
  *out = ptr;
  return IBP_OK;
}

}  // namespace

extern "C" int ibp_build_meta_noalloc(const void *rows, int64_t n_rows, int64_t row_elems,
                                      int dtype, double T, uint32_t block_elems, ibp_meta *d_meta,
                                      ibp_stream_t s) {
  size_t need = 0;
  if (int rc = ibp_meta_scratch_bytes(&need)) return rc;
  if (need > sizeof(g_noalloc_meta_counters)) return IBP_ERR_UNSUPPORTED;
  void *counters = nullptr;
  if (int rc = noalloc_counters(&counters)) return rc;
  return ibp_build_meta(rows, n_rows, row_elems, dtype, T, block_elems, d_meta, counters, s);
}
