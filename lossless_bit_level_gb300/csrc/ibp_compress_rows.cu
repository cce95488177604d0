// Compression of long rows (over 2 KiB, up to 64 KiB) for sm_103a: one CTA per row.
//
// "Reducing the GPU Memory Bottleneck with Lossless Compression for ML --
// Extended", technical summary, "Core algorithm" (compression: per-block match
// test, participation bit, invariant bits stripped, remaining bits packed) and
// "System integration" (fixed-size slot per row, GPU bitmask). Same stream as the
// warp-per-row kernels; the work of a row is spread over a whole CTA instead.
//
// A row's stream position of block j depends only on how many earlier blocks
// matched: every full block is LWB lane words of fc bits (match) or 32 bits (no
// match), so
//     offset(j) = nb + 32 * LWB * j - (32 - fc) * LWB * matched_before(j).
// With that, no scan over chunk sizes is needed. Each thread works on every
// blockDim-th 16-byte vector of the row; the CTA:
//   1. votes per vector (4 lane words against mask/bitval), folds the votes of a
//      block's GS = LWB / 4 lanes into its participation bit and ORs the bits into
//      a shared header;
//   2. one warp turns the header into per-word prefix counts of matched blocks and
//      the row's size (the formula of ibp_row_bits);
//   3. a raw row is copied out of its staging buffer; a compressed row is assembled
//      in shared memory (header words, then every vector's fields ORed in at its
//      offset: only a chunk's first and last words can be shared with a neighbour)
//      and stored with 16-byte stores.
// Rows are staged in shared memory with cp.async, the next one while the current
// one is encoded, so a CTA always has a row in flight; the stream is assembled in a
// third buffer. Each thread tests the vectors it copied itself; a barrier after the
// match pass makes the whole row visible to the pack pass.
#include <algorithm>
#include <atomic>

#include "ibp_device.cuh"
#include "ibp_internal.h"

namespace ibp {
namespace {

constexpr int ROW_THREADS = 256;
// Rows up to 64 KiB: three row buffers (two staged rows and the stream) fit in
// shared memory.
constexpr int64_t ROWS_MAX_BYTES = 64 * 1024;

struct RowArgs {
  const uint8_t *rows;
  int64_t n_rows;
  uint8_t *slots;
  int64_t slot_bytes;
  uint32_t *bitmask;
  uint32_t *row_bits;
  int32_t *status;
  const ibp_meta *meta;
  uint32_t dtype, block_elems;
  int nb, raw_words, lwt;
  int nhw;       // header words: ceil(nb / 32)
  int hdr_pad;   // header words rounded up to a multiple of 4
  int64_t raw_bytes;
};

// Stage row r into RAW with 16-byte cp.async copies (one commit group per thread).
__device__ __forceinline__ void stage_row(const RowArgs &a, int64_t r, uint32_t *RAW) {
  if (r < a.n_rows) {
    const int nvec = a.raw_words >> 2;
    const uint8_t *src = a.rows + r * a.raw_bytes;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x)
      cp_async16(reinterpret_cast<uint8_t *>(RAW) + 16 * v, src + 16 * v);
  }
  cp_async_commit();
}

// Shared memory: two staged rows, the stream buffer, two header and two prefix
// buffers and two pairs of per-row scalars (matched blocks, last block's bit).
struct RowShared {
  uint32_t *raw[2];
  uint32_t *out;
  uint32_t *hdr[2];
  uint32_t *pre[2];
  uint32_t *scal;  // [2][2]
};

template <int NR, int LWB>
__device__ void compress_rows_body(const RowArgs &a, const Code &code, const SharedRuns &sruns,
                                   const RowShared &sh) {
  constexpr int GS = LWB / 4;   // vectors (lanes) per block
  constexpr int BPS = 32 / GS;  // blocks per warp per pass
  const RegRuns<NR> runs = load_runs<NR>(sruns);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x;
  const int nvec = a.raw_words >> 2;
  const uint32_t fc = (uint32_t)code.fc;
  const uint32_t shrink = 32u - fc;
  if (blockIdx.x == 0 && tid == 0 && (a.n_rows & 31))
    atomicAnd(&a.bitmask[a.n_rows >> 5], low_mask((uint32_t)(a.n_rows & 31)));
  int64_t r = blockIdx.x;
  stage_row(a, r, sh.raw[0]);
  int par = 0;
  for (; r < a.n_rows; r += gridDim.x, par ^= 1) {
    // every thread is done with the previous row (its staged copy and the stream
    // buffer) before the next row is staged over the former
    __syncthreads();
    stage_row(a, r + gridDim.x, sh.raw[par ^ 1]);  // an empty group past the end
    cp_async_wait<1>();  // this thread's copies of row r have landed
    const uint4 *RAW4 = reinterpret_cast<const uint4 *>(sh.raw[par]);
    uint32_t *HDR = sh.hdr[par], *PRE = sh.pre[par], *S = sh.scal + 2 * par;
    for (int q = tid; q < a.nhw; q += nthr) HDR[q] = 0u;
    __syncthreads();
    // 1. participation bits (each thread tests the vectors it staged itself)
    for (int v0 = 0; v0 < nvec; v0 += nthr) {
      const int v = v0 + tid;
      bool ok = true;
      if (v < nvec) {
        const uint4 x = RAW4[v];
        ok = ((x.x & code.mask32) == code.bitval32) & ((x.y & code.mask32) == code.bitval32) &
             ((x.z & code.mask32) == code.bitval32) & ((x.w & code.mask32) == code.bitval32);
      }
      uint32_t A = __ballot_sync(FULL, ok);
#pragma unroll
      for (int sft = 1; sft < GS; sft <<= 1) A &= A >> sft;  // bit GS*j: AND of group j
      uint32_t frag = 0;
#pragma unroll
      for (int j = 0; j < BPS; ++j) frag |= ((A >> (GS * j)) & 1u) << j;
      const int b0 = (v0 + 32 * warp) / GS;
      if (b0 < a.nb) {
        if (b0 + BPS > a.nb) frag &= low_mask((uint32_t)(a.nb - b0));
        if (lane == 0 && frag) atomicOr(&HDR[b0 >> 5], frag << (b0 & 31));
      }
    }
    __syncthreads();  // the whole row has landed and the header is complete
    // 2. prefix counts of matched blocks per header word, the row's totals
    if (warp == 0) {
      uint32_t run = 0;
      for (int q0 = 0; q0 < a.nhw; q0 += 32) {
        const int q = q0 + lane;
        const uint32_t c = q < a.nhw ? (uint32_t)__popc(HDR[q]) : 0u;
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(FULL, incl, o);
          if (lane >= o) incl += y;
        }
        if (q < a.nhw) PRE[q] = run + incl - c;
        run += __shfl_sync(FULL, incl, 31);
      }
      if (lane == 0) {
        S[0] = run;
        S[1] = (HDR[(a.nb - 1) >> 5] >> ((a.nb - 1) & 31)) & 1u;
      }
    }
    __syncthreads();
    const uint32_t cnt_all = S[0], p_last = S[1];
    const uint32_t total = (uint32_t)a.nb + 32u * (uint32_t)a.raw_words -
                           shrink * ((uint32_t)LWB * cnt_all - (uint32_t)(LWB - a.lwt) * p_last);
    const uint32_t sw = (total + 31) >> 5;
    const bool comp = (int64_t)sw * 4 < a.raw_bytes;  // uniform over the CTA
    if (tid == 0) {
      if (a.row_bits) a.row_bits[r] = total;
      const uint32_t bit = 1u << (r & 31);
      if (comp) atomicOr(&a.bitmask[r >> 5], bit);
      else atomicAnd(&a.bitmask[r >> 5], ~bit);
    }
    uint4 *dst = reinterpret_cast<uint4 *>(a.slots + r * a.slot_bytes);
    if (!comp) {
      for (int v = tid; v < nvec; v += nthr) dst[v] = RAW4[v];
      continue;
    }
    // 3. the stream: header words and zeros, then every vector's fields at their offset
    const uint32_t nout4 = ((sw + 3) & ~3u) >> 2;
    uint32_t *OUT = sh.out;
    uint4 *OUT4 = reinterpret_cast<uint4 *>(OUT);
    for (uint32_t v = tid; v < nout4; v += nthr) {
      const int q = 4 * (int)v;
      OUT4[v] = make_uint4(q < a.nhw ? HDR[q] : 0u, q + 1 < a.nhw ? HDR[q + 1] : 0u,
                           q + 2 < a.nhw ? HDR[q + 2] : 0u, q + 3 < a.nhw ? HDR[q + 3] : 0u);
    }
    __syncthreads();
#pragma unroll 2
    for (int v = tid; v < nvec; v += nthr) {
      const uint4 x = RAW4[v];
      const uint32_t blk = (uint32_t)v / GS;
      const uint32_t hw = HDR[blk >> 5];
      const bool p = (hw >> (blk & 31)) & 1u;
      const uint32_t before = PRE[blk >> 5] + (uint32_t)__popc(hw & low_mask(blk & 31));
      const uint32_t F = p ? fc : 32u;
      const uint32_t pos = (uint32_t)a.nb + 32u * LWB * blk - shrink * LWB * before +
                           ((uint32_t)v - blk * GS) * 4u * F;
      uint32_t c0, c1, c2, c3;
      if (!p) {
        c0 = x.x;
        c1 = x.y;
        c2 = x.z;
        c3 = x.w;
      } else if (F == 0) {
        c0 = c1 = c2 = c3 = 0u;
      } else {
        const uint64_t f0 = extract<NR>(x.x, runs, sruns), f1 = extract<NR>(x.y, runs, sruns);
        const uint64_t f2 = extract<NR>(x.z, runs, sruns), f3 = extract<NR>(x.w, runs, sruns);
        const uint64_t lo = f0 | (f1 << F), hi = f2 | (f3 << F);  // 2F < 64 bits each
        const uint64_t w01 = lo | (hi << (2 * F));
        const uint64_t w23 = hi >> (64 - 2 * F);
        c0 = (uint32_t)w01;
        c1 = (uint32_t)(w01 >> 32);
        c2 = (uint32_t)w23;
        c3 = (uint32_t)(w23 >> 32);
      }
      const uint32_t T = 4u * F;
      if (T) {
        // words q .. q + nw - 1; only the first and the last can hold a neighbour's
        // bits (OR), the ones between belong to this chunk alone (plain stores)
        const uint32_t s = pos & 31u, q = pos >> 5;
        const uint32_t nw = (s + T + 31) >> 5;  // 1..5
        const uint32_t W1 = __funnelshift_l(c0, c1, s), W2 = __funnelshift_l(c1, c2, s);
        const uint32_t W3 = __funnelshift_l(c2, c3, s), W4 = __funnelshift_l(c3, 0u, s);
        atomicOr(&OUT[q], c0 << s);
        if (nw > 2) OUT[q + 1] = W1;
        if (nw > 3) OUT[q + 2] = W2;
        if (nw > 4) OUT[q + 3] = W3;
        if (nw > 1) atomicOr(&OUT[q + nw - 1], nw == 2 ? W1 : nw == 3 ? W2 : nw == 4 ? W3 : W4);
      }
    }
    __syncthreads();
    for (uint32_t v = tid; v < nout4; v += nthr) dst[v] = OUT4[v];
  }
  cp_async_wait<0>();
}

template <int LWB>
__global__ void __launch_bounds__(ROW_THREADS) compress_rows_kernel(RowArgs a) {
  extern __shared__ __align__(16) uint32_t smem_rows[];
  __shared__ SharedRuns sruns;
  const ibp_meta m = load_meta(a.meta);
  if (m.dtype != a.dtype || m.block_elems != a.block_elems) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(a.status, IBP_ERR_META);
    return;
  }
  const Code code = make_code(m);
  if (threadIdx.x == 0) make_runs(~code.mask32, sruns);
  RowShared sh;
  sh.raw[0] = smem_rows;  // raw_words words each, 16-byte aligned
  sh.raw[1] = sh.raw[0] + a.raw_words;
  sh.out = sh.raw[1] + a.raw_words;
  sh.hdr[0] = sh.out + a.raw_words;
  sh.hdr[1] = sh.hdr[0] + a.hdr_pad;
  sh.pre[0] = sh.hdr[1] + a.hdr_pad;
  sh.pre[1] = sh.pre[0] + a.hdr_pad;
  sh.scal = sh.pre[1] + a.hdr_pad;
  __syncthreads();
  switch (sruns.n) {
    case 0: compress_rows_body<0, LWB>(a, code, sruns, sh); break;
    case 1: compress_rows_body<1, LWB>(a, code, sruns, sh); break;
    case 2: compress_rows_body<2, LWB>(a, code, sruns, sh); break;
    case 3: compress_rows_body<3, LWB>(a, code, sruns, sh); break;
    case 4: compress_rows_body<4, LWB>(a, code, sruns, sh); break;
    default: compress_rows_body<-1, LWB>(a, code, sruns, sh); break;
  }
}

size_t rows_smem_bytes(const RowArgs &a) {
  return 4 * (3 * (size_t)a.raw_words + 4 * (size_t)a.hdr_pad + 4);
}

template <int LWB>
int launch_rows(const RowArgs &a, const DeviceInfo &dev, cudaStream_t s) {
  const size_t smem = rows_smem_bytes(a);
  static std::atomic<int> configured[64];  // the attribute is set once per device
  if (smem > 48 * 1024 && (dev.device >= 64 || !configured[dev.device].load())) {
    if (cudaFuncSetAttribute(compress_rows_kernel<LWB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dev.max_smem_optin - 2048) != cudaSuccess)
      return IBP_ERR_CUDA;
    if (dev.device < 64) configured[dev.device].store(1);
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, compress_rows_kernel<LWB>,
                                                    ROW_THREADS, smem) != cudaSuccess ||
      per_sm < 1)
    return IBP_ERR_CUDA;
  const int grid = (int)std::min<int64_t>(a.n_rows, (int64_t)dev.sm_count * per_sm);
  compress_rows_kernel<LWB><<<grid, ROW_THREADS, smem, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

}  // namespace

int64_t compress_rows_max_bytes() { return ROWS_MAX_BYTES; }

int launch_compress_rows(const void *rows, int64_t n_rows, const RowGeom &g, uint32_t dtype,
                         const ibp_meta *d_meta, void *slots, int64_t slot_bytes,
                         uint32_t *d_bitmask, uint32_t *d_row_bits, int32_t *d_status,
                         const DeviceInfo &dev, cudaStream_t s) {
  if (g.raw_words % 4 != 0 || g.raw_bytes > ROWS_MAX_BYTES) return IBP_ERR_UNSUPPORTED;
  RowArgs a;
  a.rows = static_cast<const uint8_t *>(rows);
  a.n_rows = n_rows;
  a.slots = static_cast<uint8_t *>(slots);
  a.slot_bytes = slot_bytes;
  a.bitmask = d_bitmask;
  a.row_bits = d_row_bits;
  a.status = d_status;
  a.meta = d_meta;
  a.dtype = dtype;
  a.block_elems = (uint32_t)g.B;
  a.nb = g.nb;
  a.raw_words = g.raw_words;
  a.lwt = g.lwt;
  a.nhw = (g.nb + 31) / 32;
  a.hdr_pad = (a.nhw + 3) & ~3;
  a.raw_bytes = g.raw_bytes;
  if (rows_smem_bytes(a) + 2048 > (size_t)dev.max_smem_optin) return IBP_ERR_UNSUPPORTED;
  switch (g.lwb) {
    case 8: return launch_rows<8>(a, dev, s);
    case 16: return launch_rows<16>(a, dev, s);
    case 32: return launch_rows<32>(a, dev, s);
    default: return launch_rows<64>(a, dev, s);
  }
}

}  // namespace ibp
