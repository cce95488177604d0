// Compression kernel of Invariant Bit Packing for sm_103a.
//
// "Reducing the GPU Memory Bottleneck with Lossless Compression for ML --
// Extended", technical summary, "Core algorithm" (compression: per-block match
// test against bitval, strip + shift of the invariant bits, a participation bit
// per block, run on the GPU over zero-copy memory) and "System integration"
// (fixed-size buffer per row, GPU bitmask of compressed rows).
//
// Rows of at most 2 KiB (four 512-byte steps): compress_groups_kernel below, a warp
// per group of 32 consecutive rows held in registers. Longer rows:
// compress_stream_kernel (ibp_compress_stream.cu), a warp per row in one pass.
#include <algorithm>
#include <atomic>

#include "ibp_device.cuh"
#include "ibp_internal.h"

namespace ibp {
namespace {

constexpr int COMPRESS_MAX_WARPS = 4;  // warps per CTA (measured: 3-6 % faster than 8)
constexpr int COMPRESS_CTAS_PER_SM = 6;

struct CompressArgs {
  const uint8_t *rows;
  int64_t n_rows;
  uint8_t *slots;
  int64_t slot_bytes;
  uint32_t *bitmask;
  uint32_t *row_bits;
  int32_t *status;
  const ibp_meta *meta;
  uint32_t dtype, block_elems;
  int lwb, nb, raw_words;
  int lwt;    // lane words of the last block (lwb, or fewer for a shorter tail)
  int warps;  // warps per CTA
  int64_t raw_bytes;
};

// ---------------------------------------------------------------------------
// Rows of at most 4 x 128 lane words (2 KiB): a warp owns groups of 32 consecutive
// rows. Each lane keeps its 16-byte pieces of a row in registers, the next chunk of
// rows loaded while the current one is encoded (a chunk is 4 / NSPAN rows, so eight
// 16-byte loads per lane are in flight), so the match test reads registers and raw
// rows are stored straight from them; only a compressed row's stream is assembled
// in shared memory. The group's bitmask word and its 32 row sizes are written once
// (one owner per word: no atomics).
// ---------------------------------------------------------------------------
template <int NSPAN>
__device__ __forceinline__ void load_row_regs(const CompressArgs &a, int64_t r, uint4 (&x)[NSPAN]) {
  const int lane = threadIdx.x & 31;
  const int nvec = a.raw_words / 4;
  const uint4 *src = reinterpret_cast<const uint4 *>(a.rows + r * a.raw_bytes);
#pragma unroll
  for (int i = 0; i < NSPAN; ++i) {
    const int v = 32 * i + lane;
    x[i] = (r < a.n_rows && v < nvec) ? src[v] : make_uint4(0u, 0u, 0u, 0u);
  }
}

// Encode one row held in registers; returns the size-formula bits (all lanes) and
// whether the row was stored compressed.
template <int NR, int LWB, int NSPAN>
__device__ __forceinline__ uint32_t encode_row_regs(const CompressArgs &a, const Code &code,
                                                    const RegRuns<NR> &runs,
                                                    const SharedRuns &sruns, int64_t r,
                                                    const uint4 (&x)[NSPAN], uint32_t *OUT,
                                                    bool *comp_out) {
  constexpr int GS = LWB / 4;
  constexpr int BPS = 32 / GS;
  const int lane = threadIdx.x & 31;
  const int nvec = a.raw_words / 4;
  // participation bits of at most NSPAN * BPS <= 64 blocks, kept in a register pair
  uint64_t hdr = 0;
  uint32_t cnt_all = 0;
#pragma unroll
  for (int i = 0; i < NSPAN; ++i) {
    const int v = 32 * i + lane;
    bool ok = true;
    if (v < nvec)
      ok = ((x[i].x & code.mask32) == code.bitval32) & ((x[i].y & code.mask32) == code.bitval32) &
           ((x[i].z & code.mask32) == code.bitval32) & ((x[i].w & code.mask32) == code.bitval32);
    uint32_t A = __ballot_sync(FULL, ok);
#pragma unroll
    for (int sft = 1; sft < GS; sft <<= 1) A &= A >> sft;
    uint32_t frag = 0;
#pragma unroll
    for (int j = 0; j < BPS; ++j) frag |= ((A >> (GS * j)) & 1u) << j;
    const int b0 = i * BPS;
    if (b0 >= a.nb) frag = 0;
    else if (b0 + BPS > a.nb) frag &= low_mask((uint32_t)(a.nb - b0));
    hdr |= (uint64_t)frag << b0;
    cnt_all += __popc(frag);
  }
  const uint32_t fc = (uint32_t)code.fc;
  const uint32_t shrink = 32u - fc;
  const uint32_t p_last = (uint32_t)(hdr >> (a.nb - 1)) & 1u;
  const uint32_t total = (uint32_t)a.nb + 32u * (uint32_t)a.raw_words -
                         shrink * ((uint32_t)LWB * cnt_all - (uint32_t)(LWB - a.lwt) * p_last);
  const uint32_t sw = (total + 31) >> 5;
  const bool comp = (int64_t)sw * 4 < a.raw_bytes;
  *comp_out = comp;
  uint4 *dst = reinterpret_cast<uint4 *>(a.slots + r * a.slot_bytes);
  if (!comp) {
#pragma unroll
    for (int i = 0; i < NSPAN; ++i) {
      const int v = 32 * i + lane;
      if (v < nvec) dst[v] = x[i];
    }
    return total;
  }
  const uint32_t nout = (sw + 3) & ~3u;
  for (uint32_t v = lane; v < nout / 4; v += 32)
    reinterpret_cast<uint4 *>(OUT)[v] = make_uint4(0u, 0u, 0u, 0u);
  __syncwarp();
  if (lane == 0) {
    OUT[0] = (uint32_t)hdr;
    if (a.nb > 32) OUT[1] = (uint32_t)(hdr >> 32);
  }
  __syncwarp();
  uint32_t base = (uint32_t)a.nb;
#pragma unroll
  for (int i = 0; i < NSPAN; ++i) {
    const int v = 32 * i + lane;
    const bool in = v < nvec;
    const uint32_t blk = (uint32_t)(4 * v) / LWB;
    const bool p = in && ((hdr >> blk) & 1u);
    const uint32_t F = in ? (p ? fc : 32u) : 0u;
    uint32_t c0, c1, c2, c3;
    if (!p) {
      c0 = x[i].x;
      c1 = x[i].y;
      c2 = x[i].z;
      c3 = x[i].w;
    } else if (F == 0) {
      c0 = c1 = c2 = c3 = 0u;
    } else {
      const uint64_t f0 = extract<NR>(x[i].x, runs, sruns), f1 = extract<NR>(x[i].y, runs, sruns);
      const uint64_t f2 = extract<NR>(x[i].z, runs, sruns), f3 = extract<NR>(x[i].w, runs, sruns);
      const uint64_t lo = f0 | (f1 << F), hi = f2 | (f3 << F);
      const uint64_t w01 = lo | (hi << (2 * F));
      const uint64_t w23 = hi >> (64 - 2 * F);
      c0 = (uint32_t)w01;
      c1 = (uint32_t)(w01 >> 32);
      c2 = (uint32_t)w23;
      c3 = (uint32_t)(w23 >> 32);
    }
    const uint32_t T = 4 * F;
    uint32_t incl = T;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t pos = base + incl - T;
    base += __shfl_sync(FULL, incl, 31);
    if (T) {
      const uint32_t sh = pos & 31u, q = pos >> 5;
      const uint32_t nw = (sh + T + 31) >> 5;
      atomicOr(&OUT[q], c0 << sh);
      if (nw > 1) atomicOr(&OUT[q + 1], __funnelshift_l(c0, c1, sh));
      if (nw > 2) atomicOr(&OUT[q + 2], __funnelshift_l(c1, c2, sh));
      if (nw > 3) atomicOr(&OUT[q + 3], __funnelshift_l(c2, c3, sh));
      if (nw > 4) atomicOr(&OUT[q + 4], __funnelshift_l(c3, 0u, sh));
    }
  }
  __syncwarp();
  for (uint32_t v = lane; v < nout / 4; v += 32) dst[v] = reinterpret_cast<const uint4 *>(OUT)[v];
  __syncwarp();
  return total;
}

template <int NR, int LWB, int NSPAN>
__device__ void compress_groups_body(const CompressArgs &a, const Code &code,
                                     const SharedRuns &sruns, uint32_t *OUT) {
  constexpr int CH = 4 / NSPAN;  // rows per chunk
  const RegRuns<NR> runs = load_runs<NR>(sruns);
  const int lane = threadIdx.x & 31;
  const int64_t n_groups = (a.n_rows + 31) / 32;
  const int64_t step = (int64_t)gridDim.x * a.warps;
  for (int64_t grp = (int64_t)blockIdx.x * a.warps + (threadIdx.x >> 5); grp < n_groups;
       grp += step) {
    const int64_t r0 = 32 * grp;
    const int rn = (int)min((int64_t)32, a.n_rows - r0);
    uint4 cur[CH][NSPAN], nxt[CH][NSPAN];
#pragma unroll
    for (int c = 0; c < CH; ++c) load_row_regs<NSPAN>(a, c < rn ? r0 + c : a.n_rows, cur[c]);
    uint32_t word = 0, my_bits = 0;
    for (int j0 = 0; j0 < rn; j0 += CH) {
#pragma unroll
      for (int c = 0; c < CH; ++c) {  // next chunk in flight while this one encodes
        const int j = j0 + CH + c;
        load_row_regs<NSPAN>(a, j < rn ? r0 + j : a.n_rows, nxt[c]);
      }
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int j = j0 + c;
        if (j < rn) {
          bool comp;
          const uint32_t bits =
              encode_row_regs<NR, LWB, NSPAN>(a, code, runs, sruns, r0 + j, cur[c], OUT, &comp);
          if (lane == j) my_bits = bits;
          word |= (comp ? 1u : 0u) << j;
        }
      }
#pragma unroll
      for (int c = 0; c < CH; ++c)
#pragma unroll
        for (int i = 0; i < NSPAN; ++i) cur[c][i] = nxt[c][i];
    }
    if (lane == 0) a.bitmask[grp] = word;  // bits past n_rows stay 0
    if (a.row_bits && lane < rn) a.row_bits[r0 + lane] = my_bits;
  }
}

template <int LWB, int NSPAN>
__global__ void __launch_bounds__(COMPRESS_MAX_WARPS * 32, COMPRESS_CTAS_PER_SM) compress_groups_kernel(CompressArgs a) {
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
  uint32_t *OUT = reinterpret_cast<uint32_t *>(smem) + (size_t)(threadIdx.x >> 5) * a.raw_words;
  switch (sruns.n) {
    case 0: compress_groups_body<0, LWB, NSPAN>(a, code, sruns, OUT); break;
    case 1: compress_groups_body<1, LWB, NSPAN>(a, code, sruns, OUT); break;
    case 2: compress_groups_body<2, LWB, NSPAN>(a, code, sruns, OUT); break;
    case 3: compress_groups_body<3, LWB, NSPAN>(a, code, sruns, OUT); break;
    case 4: compress_groups_body<4, LWB, NSPAN>(a, code, sruns, OUT); break;
    default: compress_groups_body<-1, LWB, NSPAN>(a, code, sruns, OUT); break;
  }
}

template <int LWB, int NSPAN>
int launch_groups(const CompressArgs &a, const DeviceInfo &dev, cudaStream_t s) {
  const size_t smem = (size_t)a.warps * 4 * a.raw_words;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, compress_groups_kernel<LWB, NSPAN>,
                                                    a.warps * 32, smem) != cudaSuccess ||
      per_sm < 1)
    return IBP_ERR_CUDA;
  const int64_t groups = (a.n_rows + 31) / 32;
  const int64_t want = (groups + a.warps - 1) / a.warps;
  const int grid = (int)std::min<int64_t>(want, (int64_t)dev.sm_count * per_sm);
  compress_groups_kernel<LWB, NSPAN><<<grid, a.warps * 32, smem, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

template <int LWB>
int launch_groups_lwb(const CompressArgs &a, const DeviceInfo &dev, int nspan, cudaStream_t s) {
  if (nspan == 1) return launch_groups<LWB, 1>(a, dev, s);
  if (nspan == 2) return launch_groups<LWB, 2>(a, dev, s);
  return launch_groups<LWB, 4>(a, dev, s);
}

}  // namespace

int launch_compress(const void *rows, int64_t n_rows, const RowGeom &g, uint32_t dtype,
                    const ibp_meta *d_meta, void *slots, int64_t slot_bytes, uint32_t *d_bitmask,
                    uint32_t *d_row_bits, int32_t *d_status, cudaStream_t s) {
  if (n_rows == 0) return IBP_OK;
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  CompressArgs a;
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
  a.lwb = g.lwb;
  a.nb = g.nb;
  a.raw_words = g.raw_words;
  a.lwt = g.lwt;
  a.raw_bytes = g.raw_bytes;
  a.warps = COMPRESS_MAX_WARPS;
  const int nspan = (g.raw_words + 127) / 128;
  if (nspan <= 4) {  // short rows: the register path
    const int ns = nspan <= 1 ? 1 : (nspan <= 2 ? 2 : 4);
    switch (g.lwb) {
      case 8: return launch_groups_lwb<8>(a, dev, ns, s);
      case 16: return launch_groups_lwb<16>(a, dev, ns, s);
      case 32: return launch_groups_lwb<32>(a, dev, ns, s);
      default: return launch_groups_lwb<64>(a, dev, ns, s);
    }
  }
  // long rows: one warp per row, one pass
  return launch_compress_stream(rows, n_rows, g, dtype, d_meta, slots, slot_bytes, d_bitmask,
                                d_row_bits, d_status, dev, s);
}

}  // namespace ibp
