// Device-side helpers shared by the IBP kernels.
//
// All kernels view a row as 32-bit "lane words": an FP32 element, two 16-bit
// elements or four 8-bit ones (the lowest-addressed element in the low bits). With
// the mask and bitval repeated across the lane word, the packed form of a lane
// word's non-invariant bits is the concatenation of its elements' fields, low
// element first -- which is exactly what the stream holds for consecutive
// elements of one block. So one code path serves every width.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ibp.h"

namespace ibp {

constexpr unsigned FULL = 0xFFFFFFFFu;
constexpr int MAX_RUNS = 16;  // a 32-bit word has at most 16 runs of ones

// Contiguous runs of non-invariant ("kept") bit positions of a lane word. Run k
// covers lane-word bits [dst, dst+len) and field bits [src, src+len), where src
// (the count of kept bits below dst) never exceeds dst. Stored as the left shift
// sh = dst - src that moves field bits to their place, the run's mask in
// lane-word space (mdst) and in field space (msrc = mdst >> sh), so one run costs
// a shift and one AND-OR to deposit or to extract.
// Built once per CTA in shared memory, then copied into registers by the
// templated bodies (NR = number of runs, known after the switch).
struct SharedRuns {
  uint32_t n;
  uint32_t sh[MAX_RUNS], mdst[MAX_RUNS], msrc[MAX_RUNS];
};

template <int NR>
struct RegRuns {
  uint32_t sh[NR > 0 ? NR : 1], mdst[NR > 0 ? NR : 1], msrc[NR > 0 ? NR : 1];
};

// Per-call code parameters derived from the metadata in device memory.
struct Code {
  uint32_t mask32;    // invariant positions, replicated to both halves for 16-bit
  uint32_t bitval32;  // their values, replicated likewise
  int fc;             // bits a lane word takes in a matching block (epw * m)
};

__device__ __forceinline__ uint32_t low_mask(uint32_t n) {  // n in [0, 32]
  return n >= 32 ? FULL : ((1u << n) - 1u);
}

// 32 bits of the 64-bit value (hi:lo) starting at bit sh (sh in [0, 31])
__device__ __forceinline__ uint32_t window(uint32_t lo, uint32_t hi, uint32_t sh) {
  return __funnelshift_r(lo, hi, sh);
}

// A w-bit pattern (w = 8, 16, 32) repeated across a 32-bit lane word.
__device__ __forceinline__ uint32_t replicate(uint32_t x, int w) {
  if (w == 8) return (x & 0xFFu) * 0x01010101u;
  if (w == 16) return (x & 0xFFFFu) * 0x00010001u;
  return x;
}

__device__ __forceinline__ int dtype_width(uint32_t dtype) {
  return dtype == IBP_FP32 ? 32 : (dtype == IBP_W8 ? 8 : 16);
}

__device__ __forceinline__ Code make_code(const ibp_meta &m) {
  Code c;
  const int w = dtype_width(m.dtype);
  c.mask32 = replicate(m.mask, w);
  c.bitval32 = replicate(m.bitval, w) & c.mask32;
  c.fc = 32 - __popc(c.mask32);
  return c;
}

// Fill the run table of `kept` (one thread).
__device__ __forceinline__ void make_runs(uint32_t kept, SharedRuns &r) {
  uint32_t n = 0, acc = 0;
  while (kept) {
    const uint32_t start = __ffs(kept) - 1;
    const uint32_t rest = kept >> start;
    const uint32_t len = (~rest == 0u) ? (32u - start) : (uint32_t)(__ffs(~rest) - 1);
    const uint32_t m = low_mask(len) << start;
    r.sh[n] = start - acc;
    r.mdst[n] = m;
    r.msrc[n] = m >> (start - acc);
    ++n;
    acc += len;
    kept &= ~m;
  }
  r.n = n;
}

template <int NR>
__device__ __forceinline__ RegRuns<NR> load_runs(const SharedRuns &s) {
  RegRuns<NR> r;
#pragma unroll
  for (int k = 0; k < NR; ++k) {
    r.sh[k] = s.sh[k];
    r.mdst[k] = s.mdst[k];
    r.msrc[k] = s.msrc[k];
  }
  return r;
}

// Spread a packed field over the kept positions of `base` (parallel bit deposit;
// base supplies the invariant bits, e.g. bitval). Field bits past the last run
// are ignored, so the field needs no masking. NR < 0: run count known only at
// run time, table read from shared memory.
template <int NR>
__device__ __forceinline__ uint32_t deposit_into(uint32_t field, uint32_t base,
                                                 const RegRuns<NR> &r, const SharedRuns &s) {
  uint32_t x = base;
  if constexpr (NR >= 0) {
#pragma unroll
    for (int k = 0; k < NR; ++k) x |= (field << r.sh[k]) & r.mdst[k];
  } else {
    for (uint32_t k = 0; k < s.n; ++k) x |= (field << s.sh[k]) & s.mdst[k];
  }
  return x;
}

// Gather the kept positions of x into a packed field (parallel bit extract).
template <int NR>
__device__ __forceinline__ uint32_t extract(uint32_t x, const RegRuns<NR> &r, const SharedRuns &s) {
  uint32_t f = 0;
  if constexpr (NR >= 0) {
#pragma unroll
    for (int k = 0; k < NR; ++k) f |= (x >> r.sh[k]) & r.msrc[k];
  } else {
    for (uint32_t k = 0; k < s.n; ++k) f |= (x >> s.sh[k]) & s.msrc[k];
  }
  return f;
}

// First error wins; nothing is written when status is null.
__device__ __forceinline__ void report(int32_t *status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ ibp_meta load_meta(const ibp_meta *m) {
  const uint4 v = __ldg(reinterpret_cast<const uint4 *>(m));
  ibp_meta r;
  r.mask = v.x;
  r.bitval = v.y;
  r.dtype = v.z;
  r.block_elems = v.w;
  return r;
}

// Asynchronous 16-byte global -> shared copy (bypasses L1); works for device
// memory and for registered host memory reached zero-copy.
// .ca: the request goes through L1, whose coalescer merges a warp's 16-byte pieces
// into whole 128-byte lines (the .cg form sends one 32-byte sector request per
// 16-byte piece, which doubles the bytes read from memory that L2 does not cache,
// such as host memory read zero-copy).
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---- mbarrier helpers ------------------------------------------------------------
// Waits are bounded: each poll asks the hardware to suspend the warp for up to
// WAIT_SUSPEND_NS (it wakes as soon as the phase completes, so a waiting warp takes
// no issue slots); a wait gives up after timeout_ns of global time (WAIT_TIMEOUT_NS
// unless a launcher passes another limit) or WAIT_POLLS polls, whichever comes
// first, and the caller then records
// IBP_ERR_TIMEOUT instead of waiting forever.
constexpr uint32_t WAIT_SUSPEND_NS = 1u << 16;
constexpr uint64_t WAIT_TIMEOUT_NS = 2000000000ull;
constexpr uint32_t WAIT_POLLS = 1u << 26;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation waits here until the kernel before it on the stream has completed
// and its memory is visible (a no-op for a kernel launched the ordinary way); a
// kernel lets the next one start launching early with launch_dependents.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(WAIT_SUSPEND_NS)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete; gives up when the
// time or poll bound runs out, or as soon as *abort (nullable) is set. Returns true
// when the phase completed.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const volatile int *abort,
                                          uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < WAIT_POLLS; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((abort && *abort) || global_ns() - t0 > timeout_ns) return false;
  }
  return false;
}

// Make `bar` track this thread's cp.async copies issued so far: the pending count
// of the current phase is raised by one now and lowered when those copies have
// landed, so the phase cannot complete before them.
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

}  // namespace ibp
