// Decompress-gather kernel of Invariant Bit Packing for sm_103a.
//
// "Reducing the GPU Memory Bottleneck with Lossless Compression for ML --
// Extended", technical summary, "Core algorithm" (decompression) and "System
// integration" (fixed-size buffers of which only the compressed part is read,
// GPU-resident bitmask of compressed rows).
//
// Work unit: one segment (at most 32 consecutive blocks) of one requested row.
// Each warp takes a group of G units at a time:
//   1. header stage, one lane per unit: index -> bitmask bit -> participation
//      bits of the row header. Population counts of the header words give the
//      number of compressed blocks before the segment, and with it the
//      segment's first bit (the prefix scan of block sizes reduces to a popcount
//      because a block is either B*m or B*w bits long);
//   2. staging: the warp copies exactly the 16-byte-aligned span of the slot that
//      holds the segment into shared memory with cp.async (16 B per lane per
//      step, coalesced; works for HBM and for registered host memory reached
//      zero-copy over the host link);
//   3. decode: each lane rebuilds 4 lane words (16 output bytes) per step: block
//      of the vector, its participation bit, popcount of the earlier bits in the
//      segment -> bit position; funnel-shift the field out of shared memory,
//      deposit it over the non-invariant positions, OR bitval, 128-bit store.
#include <algorithm>

#include "ibp_device.cuh"
#include "ibp_internal.h"

namespace ibp {
namespace {

constexpr int GATHER_WARPS = 8;         // warps per CTA
constexpr int SEG_TARGET_BYTES = 4096;  // raw bytes per segment (at most 32 blocks)
constexpr int WARP_SMEM_TARGET = 6144;  // staging bytes per warp

struct GatherArgs {
  const uint8_t *slots;
  int64_t slot_bytes;
  int64_t n_rows;
  const uint32_t *bitmask;
  const ibp_meta *meta;
  const int64_t *idx;
  int64_t n_idx;
  uint32_t *out;
  int32_t *status;
  uint32_t dtype, block_elems;
  int lwb, lwb_shift, nb, raw_words;
  int seg_blocks, nseg;
  int units_per_group;  // G
  int unit_bytes;       // shared staging bytes per unit
  int64_t n_units, n_groups;
  int64_t raw_bytes;
};

// What the header stage learns about a unit (held by the lane of that unit).
struct Unit {
  const uint8_t *src;  // first staged byte
  int64_t out_word;    // first output lane word of the segment
  uint32_t nchunk;     // 16-byte chunks to stage
  uint32_t lsb;        // bit offset of the segment's first block in the staged bytes
  uint32_t segp;       // participation bits of the segment's blocks
  uint32_t nblk;       // blocks in the segment
  uint32_t kind;       // 0 skip, 1 raw row, 2 compressed row
};

__device__ __forceinline__ Unit header_stage(const GatherArgs &a, const Code &code, int64_t u) {
  Unit un;
  un.kind = 0;
  un.src = nullptr;
  un.out_word = 0;
  un.nchunk = 0;
  un.lsb = 0;
  un.segp = 0;
  un.nblk = 0;
  if (u >= a.n_units) return un;
  const int64_t i = u / a.nseg;
  const int s = (int)(u - i * a.nseg);
  const int64_t r = a.idx[i];
  const int b0 = s * a.seg_blocks;
  const int nblk = min(a.seg_blocks, a.nb - b0);
  un.nblk = nblk;
  un.out_word = i * (int64_t)a.raw_words + (int64_t)b0 * a.lwb;
  if (r < 0 || r >= a.n_rows) {
    report(a.status, IBP_ERR_INDEX);
    return un;
  }
  const uint8_t *slot = a.slots + r * a.slot_bytes;
  const bool comp = (a.bitmask[r >> 5] >> (r & 31)) & 1u;
  if (!comp) {
    un.kind = 1;
    un.src = slot + (size_t)b0 * a.lwb * 4;
    un.nchunk = (uint32_t)(nblk * a.lwb / 4);
    return un;
  }
  // participation bits: nb bits at the start of the slot
  const uint32_t *hw = reinterpret_cast<const uint32_t *>(slot);
  const int nhw = (a.nb + 31) >> 5;
  uint32_t cnt_all = 0, cnt0 = 0;
  for (int q = 0; q < nhw; ++q) {
    uint32_t word = hw[q];
    if (q == nhw - 1) word &= low_mask((uint32_t)(a.nb - 32 * q));
    const uint32_t c = __popc(word);
    cnt_all += c;
    if (32 * q + 32 <= b0) cnt0 += c;
    else if (32 * q < b0) cnt0 += __popc(word & low_mask((uint32_t)(b0 - 32 * q)));
  }
  const int q0 = b0 >> 5;
  const uint32_t lo = hw[q0];
  const uint32_t hi = (q0 + 1 < nhw) ? hw[q0 + 1] : 0u;
  const uint32_t segp = window(lo, hi, (uint32_t)(b0 & 31)) & low_mask((uint32_t)nblk);
  const uint32_t shrink = (uint32_t)(32 - code.fc);  // bits a lane word loses in a matching block
  const uint32_t total = (uint32_t)a.nb + (uint32_t)a.lwb * (32u * (uint32_t)a.nb - shrink * cnt_all);
  const uint32_t words = (total + 31) >> 5;
  if ((int64_t)words * 4 >= a.raw_bytes) {
    report(a.status, IBP_ERR_CORRUPT);
    return un;
  }
  const uint32_t st = (uint32_t)a.nb + (uint32_t)a.lwb * (32u * (uint32_t)b0 - shrink * cnt0);
  const uint32_t en = st + (uint32_t)a.lwb * (32u * (uint32_t)nblk - shrink * __popc(segp));
  const uint32_t w0 = (st >> 5) & ~3u;
  const uint32_t w1 = ((en + 127) >> 7) << 2;
  un.kind = 2;
  un.src = slot + (size_t)w0 * 4;
  un.nchunk = (w1 - w0) >> 2;
  un.lsb = st - 32 * w0;
  un.segp = segp;
  return un;
}

template <int NR>
__device__ __forceinline__ uint32_t rebuild(uint32_t x, bool p, const Code &c,
                                            const RegRuns<NR> &runs, const SharedRuns &sruns) {
  return p ? (deposit<NR>(x, runs, sruns) | c.bitval32) : x;
}

template <int NR>
__device__ void gather_body(const GatherArgs &a, const Code &code, const SharedRuns &sruns,
                            uint8_t *warp_smem) {
  const RegRuns<NR> runs = load_runs<NR>(sruns);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int G = a.units_per_group;
  const uint32_t fc = (uint32_t)code.fc;
  const uint32_t fc_mask = low_mask(fc);
  const uint32_t shrink = 32u - fc;

  for (int64_t grp = (int64_t)blockIdx.x * GATHER_WARPS + warp; grp < a.n_groups;
       grp += (int64_t)gridDim.x * GATHER_WARPS) {
    // 1. header stage: lane j < G handles unit grp*G + j
    Unit un;
    if (lane < G) un = header_stage(a, code, grp * G + lane);
    else un = header_stage(a, code, a.n_units);  // empty

    // 2. staging
    for (int j = 0; j < G; ++j) {
      const uint32_t kind = __shfl_sync(FULL, un.kind, j);
      if (kind == 0) continue;
      const uint8_t *src = reinterpret_cast<const uint8_t *>(
          __shfl_sync(FULL, reinterpret_cast<unsigned long long>(un.src), j));
      const uint32_t n = __shfl_sync(FULL, un.nchunk, j);
      uint8_t *dst = warp_smem + j * a.unit_bytes;
      for (uint32_t c = lane; c < n; c += 32) cp_async16(dst + 16 * c, src + 16 * c);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncwarp();

    // 3. decode
    for (int j = 0; j < G; ++j) {
      const uint32_t kind = __shfl_sync(FULL, un.kind, j);
      if (kind == 0) continue;
      const int64_t out_word = __shfl_sync(FULL, un.out_word, j);
      const uint32_t nblk = __shfl_sync(FULL, un.nblk, j);
      const uint32_t nvec = nblk * (uint32_t)a.lwb / 4;
      const uint32_t *S = reinterpret_cast<const uint32_t *>(warp_smem + j * a.unit_bytes);
      uint4 *dst = reinterpret_cast<uint4 *>(a.out + out_word);
      if (kind == 1) {
        const uint4 *S4 = reinterpret_cast<const uint4 *>(S);
        for (uint32_t v = lane; v < nvec; v += 32) dst[v] = S4[v];
        continue;
      }
      const uint32_t lsb = __shfl_sync(FULL, un.lsb, j);
      const uint32_t segp = __shfl_sync(FULL, un.segp, j);
      for (uint32_t v = lane; v < nvec; v += 32) {
        const uint32_t lw = 4 * v;
        const uint32_t lb = lw >> a.lwb_shift;
        const bool p = (segp >> lb) & 1u;
        const uint32_t cnt = __popc(segp & low_mask(lb));
        const uint32_t f = p ? fc : 32u;
        const uint32_t fm = p ? fc_mask : FULL;
        uint32_t pos = lsb + (uint32_t)a.lwb * (32u * lb - shrink * cnt) +
                       (lw - (lb << a.lwb_shift)) * f;
        uint32_t y[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint32_t q = pos >> 5;
          const uint32_t x = window(S[q], S[q + 1], pos & 31) & fm;
          y[t] = rebuild<NR>(x, p, code, runs, sruns);
          pos += f;
        }
        dst[v] = make_uint4(y[0], y[1], y[2], y[3]);
      }
    }
    __syncwarp();
  }
}

__global__ void __launch_bounds__(GATHER_WARPS * 32) gather_kernel(GatherArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ SharedRuns sruns;
  const ibp_meta m = load_meta(a.meta);
  if (m.dtype != a.dtype || m.block_elems != a.block_elems) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(a.status, IBP_ERR_META);
    return;
  }
  const Code code = make_code(m);
  if (threadIdx.x == 0) make_runs(~code.mask32, sruns);
  __syncthreads();
  uint8_t *warp_smem = smem + (threadIdx.x >> 5) * (a.units_per_group * a.unit_bytes);
  switch (sruns.n) {
    case 0: gather_body<0>(a, code, sruns, warp_smem); break;
    case 1: gather_body<1>(a, code, sruns, warp_smem); break;
    case 2: gather_body<2>(a, code, sruns, warp_smem); break;
    case 3: gather_body<3>(a, code, sruns, warp_smem); break;
    case 4: gather_body<4>(a, code, sruns, warp_smem); break;
    default: gather_body<-1>(a, code, sruns, warp_smem); break;
  }
}

int ilog2(int x) {
  int s = 0;
  while ((1 << s) < x) ++s;
  return s;
}

}  // namespace

int launch_gather(const void *slots, int64_t slot_bytes, int64_t n_rows, const RowGeom &g,
                  uint32_t dtype, const uint32_t *d_bitmask, const ibp_meta *d_meta,
                  const int64_t *d_idx, int64_t n_idx, void *out, int32_t *d_status,
                  cudaStream_t s) {
  if (n_idx == 0) return IBP_OK;
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  GatherArgs a;
  a.slots = static_cast<const uint8_t *>(slots);
  a.slot_bytes = slot_bytes;
  a.n_rows = n_rows;
  a.bitmask = d_bitmask;
  a.meta = d_meta;
  a.idx = d_idx;
  a.n_idx = n_idx;
  a.out = static_cast<uint32_t *>(out);
  a.status = d_status;
  a.dtype = dtype;
  a.block_elems = (uint32_t)g.B;
  a.lwb = g.lwb;
  a.lwb_shift = ilog2(g.lwb);
  a.nb = g.nb;
  a.raw_words = g.raw_words;
  const int block_bytes = g.lwb * 4;
  a.seg_blocks = std::max(1, std::min({g.nb, 32, SEG_TARGET_BYTES / block_bytes}));
  a.nseg = (g.nb + a.seg_blocks - 1) / a.seg_blocks;
  a.unit_bytes = a.seg_blocks * block_bytes + 64;
  a.units_per_group = std::max(1, std::min(8, WARP_SMEM_TARGET / a.unit_bytes));
  a.n_units = n_idx * a.nseg;
  a.n_groups = (a.n_units + a.units_per_group - 1) / a.units_per_group;
  a.raw_bytes = g.raw_bytes;
  const size_t smem = (size_t)GATHER_WARPS * a.units_per_group * a.unit_bytes;
  static int configured[64] = {0};
  if (dev.device < 64 && !configured[dev.device]) {
    if (cudaFuncSetAttribute(gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dev.max_smem_optin - (int)sizeof(SharedRuns) - 1024) != cudaSuccess)
      return IBP_ERR_CUDA;
    configured[dev.device] = 1;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gather_kernel, GATHER_WARPS * 32,
                                                    smem) != cudaSuccess ||
      per_sm < 1)
    return IBP_ERR_CUDA;
  const int64_t want = (a.n_groups + GATHER_WARPS - 1) / GATHER_WARPS;
  const int grid = (int)std::min<int64_t>(want, (int64_t)dev.sm_count * per_sm);
  gather_kernel<<<grid, GATHER_WARPS * 32, smem, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

}  // namespace ibp
