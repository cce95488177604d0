// Compression kernel of Invariant Bit Packing for sm_103a.
//
// "Reducing the GPU Memory Bottleneck with Lossless Compression for ML --
// Extended", technical summary, "Core algorithm" (compression: per-block match
// test against bitval, strip + shift of the invariant bits, a participation bit
// per block, run on the GPU over zero-copy memory) and "System integration"
// (fixed-size buffer per row, GPU bitmask of compressed rows).
//
// One warp encodes one row; a CTA owns 32 consecutive rows so that it writes
// whole bitmask words (no atomics, deterministic). Per row:
//   a. the raw row is staged in shared memory with 128-bit loads (read once,
//      also when it sits in host memory);
//   b. match pass: lane-strided lane words, ballot per 32 lane words -> the
//      participation bit of each block -> header words; the compressed-block
//      count gives the row's exact size and the raw-or-compressed decision;
//   c. pack pass (compressed rows only): per 32 lane words each lane extracts
//      its field; the lane that owns payload word t collects the fields that
//      overlap it with shuffles (each word is built by one lane, no atomics);
//      the payload is shifted past the nb header bits with a carry word and
//      written to a shared-memory copy of the stream;
//   d. the stream (or the raw row) is written to the slot with 128-bit stores.
#include <algorithm>

#include "ibp_device.cuh"
#include "ibp_internal.h"

namespace ibp {
namespace {

constexpr int COMPRESS_MAX_WARPS = 8;
constexpr int COMPRESS_SMEM_BUDGET = 200 * 1024;

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
  int lwb, lwb_shift, nb, raw_words;
  int warps;
  int warp_bytes;  // shared bytes per warp
  int hdr_words;   // header words reserved per warp (multiple of 4)
  int64_t n_units; // ceil(n_rows / 32)
  int64_t raw_bytes;
};

// Pack one 32-lane-word chunk. Lane l holds value v of width F_l bits, where
// all lanes of a segment share one width (one segment of 32 lanes, or two of 16
// when a block is 16 lane words). Returns the payload word owned by this lane
// (valid for lane < *nwords).
__device__ __forceinline__ uint32_t pack_chunk(uint32_t v, uint32_t F, bool two_seg,
                                               uint32_t *nwords) {
  const int lane = threadIdx.x & 31;
  uint32_t F0, F1, n0, n1;
  if (two_seg) {
    F0 = __shfl_sync(FULL, F, 0);
    F1 = __shfl_sync(FULL, F, 16);
    n0 = F0 >> 1;  // 16 lanes * F bits / 32
    n1 = F1 >> 1;
  } else {
    F0 = F;  // uniform
    F1 = 0;
    n0 = F0;
    n1 = 0;
  }
  *nwords = n0 + n1;
  uint32_t Fmin = 32;
  if (F0 > 0) Fmin = min(Fmin, F0);
  if (F1 > 0) Fmin = min(Fmin, F1);
  if (n0 + n1 == 0) return 0;
  const uint32_t K = (32 + Fmin - 1) / Fmin + 1;
  // this lane's segment
  uint32_t t = (uint32_t)lane, base = 0, Fs = F0, seg_lanes = two_seg ? 16u : 32u;
  if ((uint32_t)lane >= n0) {
    t = (uint32_t)lane - n0;
    base = 16;
    Fs = F1;
  }
  const bool owner = (uint32_t)lane < n0 + n1 && Fs > 0;
  const uint32_t l0 = owner ? base + (32 * t) / Fs : 0;
  uint32_t P = 0;
  for (uint32_t it = 0; it < K; ++it) {
    const uint32_t l = l0 + it;
    const uint32_t vl = __shfl_sync(FULL, v, (int)min(l, 31u));
    if (owner && l < base + seg_lanes) {
      const int shift = (int)((l - base) * Fs) - (int)(32 * t);
      if (shift < 32 && shift > -(int)Fs) P |= shift >= 0 ? (vl << shift) : (vl >> (-shift));
    }
  }
  return P;
}

template <int NR>
__device__ bool compress_row(const CompressArgs &a, const Code &code, const RegRuns<NR> &runs,
                             const SharedRuns &sruns, int64_t r, uint32_t *RAW, uint32_t *OUT,
                             uint32_t *HDR) {
  const int lane = threadIdx.x & 31;
  const int nvec = a.raw_words / 4;
  // a. stage the raw row
  const uint4 *src = reinterpret_cast<const uint4 *>(a.rows + r * a.raw_bytes);
  for (int v = lane; v < nvec; v += 32) reinterpret_cast<uint4 *>(RAW)[v] = src[v];
  __syncwarp();

  // b. participation bits
  const int nchunks = a.raw_words / 32 + ((a.raw_words & 31) ? 1 : 0);
  uint32_t hacc = 0, cnt_all = 0, pair_ok = 1;
  for (int c = 0; c < nchunks; ++c) {
    const int lw = 32 * c + lane;
    const bool in = lw < a.raw_words;
    const uint32_t x = in ? RAW[lw] : code.bitval32;
    const uint32_t M = __ballot_sync(FULL, (x & code.mask32) == code.bitval32);
    uint32_t bits, nbits, b;
    if (a.lwb == 16) {
      b = 2 * c;
      bits = ((M & 0xFFFFu) == 0xFFFFu ? 1u : 0u) | ((M >> 16) == 0xFFFFu ? 2u : 0u);
      nbits = 2;
    } else if (a.lwb == 32) {
      b = c;
      bits = M == FULL ? 1u : 0u;
      nbits = 1;
    } else {  // 64: two chunks per block
      if ((c & 1) == 0) {
        pair_ok = M == FULL;
        continue;
      }
      b = c >> 1;
      bits = (pair_ok && M == FULL) ? 1u : 0u;
      nbits = 1;
    }
    if (b + nbits > (uint32_t)a.nb) {  // half-used last chunk (16-lane-word blocks)
      nbits = (uint32_t)a.nb - b;
      bits &= low_mask(nbits);
    }
    hacc |= bits << (b & 31);
    cnt_all += __popc(bits);
    const uint32_t last = b + nbits - 1;
    if ((last & 31) == 31 || last == (uint32_t)a.nb - 1) {
      if (lane == 0) HDR[b >> 5] = hacc;
      hacc = 0;
    }
  }
  const uint32_t shrink = 32u - (uint32_t)code.fc;
  const uint32_t total = (uint32_t)a.nb + (uint32_t)a.lwb * (32u * (uint32_t)a.nb - shrink * cnt_all);
  const uint32_t sw = (total + 31) >> 5;
  const bool comp = (int64_t)sw * 4 < a.raw_bytes;
  if (a.row_bits && lane == 0) a.row_bits[r] = total;
  __syncwarp();

  uint4 *dst = reinterpret_cast<uint4 *>(a.slots + r * a.slot_bytes);
  if (!comp) {
    for (int v = lane; v < nvec; v += 32) dst[v] = reinterpret_cast<const uint4 *>(RAW)[v];
    return false;
  }

  // c. pack
  const uint32_t nbw = (uint32_t)a.nb >> 5, sh = (uint32_t)a.nb & 31u;
  for (uint32_t q = lane; q < nbw; q += 32) OUT[q] = HDR[q];
  uint32_t carry = sh ? HDR[nbw] : 0u;  // low sh bits of the partly filled word
  uint32_t off = nbw;
  const bool two_seg = a.lwb == 16;
  for (int c = 0; c < nchunks; ++c) {
    const int lw = 32 * c + lane;
    const bool in = lw < a.raw_words;
    const uint32_t x = in ? RAW[lw] : 0u;
    const uint32_t b = (uint32_t)lw >> a.lwb_shift;
    const bool p = in && ((HDR[b >> 5] >> (b & 31)) & 1u);
    const uint32_t F = in ? (p ? (uint32_t)code.fc : 32u) : 0u;
    const uint32_t v = p ? extract<NR>(x, runs, sruns) : x;
    uint32_t nw;
    const uint32_t P = pack_chunk(v, F, two_seg, &nw);
    if (nw == 0) continue;
    if (sh == 0) {
      if ((uint32_t)lane < nw) OUT[off + lane] = P;
    } else {
      const uint32_t prev = __shfl_up_sync(FULL, P, 1);
      const uint32_t lo = lane == 0 ? carry : (prev >> (32 - sh));
      if ((uint32_t)lane < nw) OUT[off + lane] = (P << sh) | lo;
      carry = __shfl_sync(FULL, P, (int)nw - 1) >> (32 - sh);
    }
    off += nw;
  }
  if (sh && lane == 0) OUT[off] = carry;
  // zero the tail of the last 16-byte vector
  const uint32_t nout = (sw + 3) & ~3u;
  if ((uint32_t)lane < nout - sw) OUT[sw + lane] = 0u;
  __syncwarp();
  // d. store the stream
  for (uint32_t v = lane; v < nout / 4; v += 32) dst[v] = reinterpret_cast<const uint4 *>(OUT)[v];
  return true;
}

template <int NR>
__device__ void compress_body(const CompressArgs &a, const Code &code, const SharedRuns &sruns,
                              uint8_t *smem, uint32_t *flags) {
  const RegRuns<NR> runs = load_runs<NR>(sruns);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  uint8_t *mine = smem + (size_t)warp * a.warp_bytes;
  uint32_t *HDR = reinterpret_cast<uint32_t *>(mine);
  uint32_t *RAW = HDR + a.hdr_words;
  uint32_t *OUT = RAW + a.raw_words;
  for (int64_t unit = blockIdx.x; unit < a.n_units; unit += gridDim.x) {
    for (int k = warp; k < 32; k += a.warps) {
      const int64_t r = unit * 32 + k;
      bool comp = false;
      if (r < a.n_rows) comp = compress_row<NR>(a, code, runs, sruns, r, RAW, OUT, HDR);
      if (lane == 0) flags[k] = comp ? 1u : 0u;
      __syncwarp();
    }
    __syncthreads();
    if (warp == 0) {
      const uint32_t word = __ballot_sync(FULL, flags[lane] != 0);
      if (lane == 0) a.bitmask[unit] = word;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(COMPRESS_MAX_WARPS * 32) compress_kernel(CompressArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ SharedRuns sruns;
  __shared__ uint32_t flags[32];
  const ibp_meta m = load_meta(a.meta);
  if (m.dtype != a.dtype || m.block_elems != a.block_elems) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(a.status, IBP_ERR_META);
    return;
  }
  const Code code = make_code(m);
  if (threadIdx.x == 0) make_runs(~code.mask32, sruns);
  __syncthreads();
  switch (sruns.n) {
    case 0: compress_body<0>(a, code, sruns, smem, flags); break;
    case 1: compress_body<1>(a, code, sruns, smem, flags); break;
    case 2: compress_body<2>(a, code, sruns, smem, flags); break;
    case 3: compress_body<3>(a, code, sruns, smem, flags); break;
    case 4: compress_body<4>(a, code, sruns, smem, flags); break;
    default: compress_body<-1>(a, code, sruns, smem, flags); break;
  }
}

int ilog2(int x) {
  int s = 0;
  while ((1 << s) < x) ++s;
  return s;
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
  a.lwb_shift = ilog2(g.lwb);
  a.nb = g.nb;
  a.raw_words = g.raw_words;
  a.raw_bytes = g.raw_bytes;
  a.hdr_words = (((g.nb + 31) / 32) + 3) & ~3;
  // header + raw row + stream (never longer than the raw row when kept)
  a.warp_bytes = 4 * (a.hdr_words + 2 * g.raw_words);
  const int limit = std::min(COMPRESS_SMEM_BUDGET, dev.max_smem_optin - 2048);
  a.warps = std::min(COMPRESS_MAX_WARPS, limit / a.warp_bytes);
  if (a.warps < 1) return IBP_ERR_UNSUPPORTED;
  a.n_units = (n_rows + 31) / 32;
  const size_t smem = (size_t)a.warps * a.warp_bytes;
  static int configured[64] = {0};
  if (dev.device < 64 && !configured[dev.device]) {
    if (cudaFuncSetAttribute(compress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             limit) != cudaSuccess)
      return IBP_ERR_CUDA;
    configured[dev.device] = 1;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, compress_kernel, a.warps * 32,
                                                    smem) != cudaSuccess ||
      per_sm < 1)
    return IBP_ERR_CUDA;
  const int grid = (int)std::min<int64_t>(a.n_units, (int64_t)dev.sm_count * per_sm);
  compress_kernel<<<grid, a.warps * 32, smem, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

}  // namespace ibp
