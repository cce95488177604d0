// Per-position metadata variant of Invariant Bit Packing for sm_103a.
//
// "Reducing the GPU Memory Bottleneck with Lossless Compression for ML --
// Extended", technical summary, "Core algorithm": the metadata is a mask/bitval
// kept in GPU memory, "kilobyte-scale". Read as one pair per element position of a
// row, each position (a feature column, an embedding dimension) gets its own
// invariant bits: the preprocessing rule applied to element e of every row. A
// block matches when each element holds its own position's bitval; a matching
// element is stored as a field of w - popcount(mask_e) bits. Everything else (the
// participation bits first, LSB-first words, the store rule) is the shared-mask
// format.
//
// Lane words: lane word k of a row holds elements k*epw .. k*epw + epw - 1, so its
// mask M[k] and bitval V[k] are those positions' masks side by side, and its field
// in a matching block is the concatenation of the elements' fields (F[k] =
// 32 - popcount(M[k]) bits). Every kernel derives, in shared memory, per lane word
// M, V, F and OFF (the bit offset of its field inside its block), and per block
// FB (the block's bits when it matches), from the per-position arrays.
// Kernels:
//   pos_count_kernel / pos_finalize_kernel: per-column positional popcount (a
//     thread per (lane-word column, row range), bit-sliced carry-save counters,
//     64-bit atomics per column) and the threshold rule per position;
//   pos_compress_kernel: a warp per row (rows grid-strided, the next row staged
//     with cp.async), match test per lane word against its own M/V, block bits by
//     ballot, row size from FB, fields extracted and packed with a warp scan;
//   pos_gather_kernel: a warp per requested row, the slot's raw-size prefix staged
//     (double-buffered, the next row's copy in flight during decode), block offsets
//     by a warp scan of block sizes, each lane word rebuilt from its field.
// Parallel bit extract/deposit walk the runs of a lane word's kept bits (a few per
// word for float masks), since each position has its own mask.
#include <algorithm>

#include "ibp_device.cuh"
#include "ibp_internal.h"
#include "ibp_popcount.cuh"

namespace ibp {
namespace {

constexpr int POS_THREADS = 256;
constexpr int POS_WARPS = POS_THREADS / 32;
constexpr int POS_SMEM_BUDGET = 200 * 1024;

// ---------------------------------------------------------------- bit runs
// The set bits of `kept`, as runs [start, start + len): deposit puts consecutive
// field bits into them in ascending order, extract takes them out.
__device__ __forceinline__ uint32_t deposit_runs(uint32_t field, uint32_t kept) {
  uint32_t x = 0, used = 0;
  while (kept) {
    const uint32_t start = __ffs(kept) - 1;
    const uint32_t rest = kept >> start;
    const uint32_t len = (~rest == 0u) ? 32u - start : (uint32_t)(__ffs(~rest) - 1);
    const uint32_t m = low_mask(len) << start;
    x |= (field << (start - used)) & m;
    used += len;
    kept &= ~m;
  }
  return x;
}

__device__ __forceinline__ uint32_t extract_runs(uint32_t x, uint32_t kept) {
  uint32_t f = 0, used = 0;
  while (kept) {
    const uint32_t start = __ffs(kept) - 1;
    const uint32_t rest = kept >> start;
    const uint32_t len = (~rest == 0u) ? 32u - start : (uint32_t)(__ffs(~rest) - 1);
    const uint32_t m = low_mask(len) << start;
    f |= (x & m) >> (start - used);
    used += len;
    kept &= ~m;
  }
  return f;
}

// ---------------------------------------------------------------- tables
struct Geo {
  int w, lwb, lwb_shift, lwt, nb, raw_words;
};

struct Tables {
  uint32_t *M, *V, *FB;
  uint16_t *OFF;
  uint8_t *F;
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

__host__ __device__ inline size_t table_bytes(int raw_words, int nb) {
  return 2 * align16(4 * (size_t)raw_words) + align16(4 * (size_t)nb) +
         align16(2 * (size_t)raw_words) + align16((size_t)raw_words);
}

__device__ inline Tables carve_tables(uint8_t *base, const Geo &g) {
  Tables t;
  t.M = reinterpret_cast<uint32_t *>(base);
  base += align16(4 * (size_t)g.raw_words);
  t.V = reinterpret_cast<uint32_t *>(base);
  base += align16(4 * (size_t)g.raw_words);
  t.FB = reinterpret_cast<uint32_t *>(base);
  base += align16(4 * (size_t)g.nb);
  t.OFF = reinterpret_cast<uint16_t *>(base);
  base += align16(2 * (size_t)g.raw_words);
  t.F = base;
  return t;
}

// All threads of the CTA; ends with a barrier.
__device__ void build_tables(const uint32_t *pmask, const uint32_t *pbitval, const Geo &g,
                             const Tables &t) {
  const int epw = 32 / g.w;
  const uint32_t wm = low_mask((uint32_t)g.w);
  for (int k = threadIdx.x; k < g.raw_words; k += blockDim.x) {
    uint32_t m = 0, v = 0;
    for (int i = 0; i < epw; ++i) {
      const uint32_t mk = __ldg(pmask + k * epw + i) & wm;
      m |= mk << (i * g.w);
      v |= (__ldg(pbitval + k * epw + i) & mk) << (i * g.w);
    }
    t.M[k] = m;
    t.V[k] = v;
    t.F[k] = (uint8_t)(32 - __popc(m));
  }
  __syncthreads();
  for (int b = threadIdx.x; b < g.nb; b += blockDim.x) {
    const int k0 = b * g.lwb;
    const int k1 = min(k0 + g.lwb, g.raw_words);
    uint32_t s = 0;
    for (int k = k0; k < k1; ++k) {
      t.OFF[k] = (uint16_t)s;
      s += t.F[k];
    }
    t.FB[b] = s;
  }
  __syncthreads();
}

// lane words of block b (the last may be shorter)
__device__ __forceinline__ uint32_t block_words(const Geo &g, int b) {
  return (uint32_t)(b == g.nb - 1 ? g.lwt : g.lwb);
}

// ---------------------------------------------------------------- metadata
__global__ void __launch_bounds__(POS_THREADS)
    pos_count_kernel(const uint32_t *__restrict__ rows, int64_t n_rows, int raw_words,
                     int64_t rows_per_chunk, int64_t n_chunks, unsigned long long *counters) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)raw_words * n_chunks) return;
  const int k = (int)(t % raw_words);
  const int64_t chunk = t / raw_words;
  const int64_t r0 = chunk * rows_per_chunk;
  const int64_t r1 = min(n_rows, r0 + rows_per_chunk);
  Planes P;
#pragma unroll
  for (int j = 0; j < 32; ++j) P.tot[j] = 0;
  int steps = 0;
  for (int64_t r = r0; r < r1; r += 8) {
    uint32_t x[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) x[q] = (r + q < r1) ? __ldg(rows + (r + q) * raw_words + k) : 0u;
    add8(P, make_uint4(x[0], x[1], x[2], x[3]), make_uint4(x[4], x[5], x[6], x[7]));
    if (++steps == 255) {
      flush_eights(P);
      steps = 0;
    }
  }
  flush_eights(P);
  fold_planes(P);
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (P.tot[j]) atomicAdd(&counters[(int64_t)k * 32 + j], (unsigned long long)P.tot[j]);
}

__global__ void pos_finalize_kernel(const unsigned long long *counters, int64_t n_rows,
                                    int row_elems, int w, double T, uint32_t *pmask,
                                    uint32_t *pbitval) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= row_elems) return;
  const int epw = 32 / w;
  const int64_t base = (int64_t)(p / epw) * 32 + (p % epw) * w;
  const unsigned long long N = (unsigned long long)n_rows;
  uint32_t mask = 0, bitval = 0;
  for (int j = 0; j < w; ++j) {
    const unsigned long long c1 = counters[base + j];
    const unsigned long long c0 = N - c1;
    const bool v = c1 > c0;  // a tie keeps 0
    const unsigned long long held = v ? c1 : c0;
    if ((double)held >= T * (double)N) {
      mask |= 1u << j;
      bitval |= (uint32_t)v << j;
    }
  }
  pmask[p] = mask;
  pbitval[p] = bitval;
}

// Block-position metadata: position q of a block takes the rule over the counts of
// every element position e with e % B == q (the element at position q of every
// block of every row; a shorter last block contributes only the positions it has),
// then every element position gets its block position's pair. One CTA.
__global__ void pos_block_finalize_kernel(const unsigned long long *counters, int64_t n_rows,
                                          int row_elems, int w, int B, double T,
                                          uint32_t *pmask, uint32_t *pbitval) {
  __shared__ uint32_t qmask[64], qbitval[64];
  const int q = threadIdx.x;
  const int epw = 32 / w;
  if (q < B && q < row_elems) {
    const int64_t copies = (row_elems - q + B - 1) / B;  // blocks that have position q
    const unsigned long long N = (unsigned long long)(n_rows * copies);
    uint32_t mask = 0, bitval = 0;
    for (int j = 0; j < w; ++j) {
      unsigned long long c1 = 0;
      for (int e = q; e < row_elems; e += B)
        c1 += counters[(int64_t)(e / epw) * 32 + (e % epw) * w + j];
      const unsigned long long c0 = N - c1;
      const bool v = c1 > c0;  // a tie keeps 0
      const unsigned long long held = v ? c1 : c0;
      if ((double)held >= T * (double)N) {
        mask |= 1u << j;
        bitval |= (uint32_t)v << j;
      }
    }
    qmask[q] = mask;
    qbitval[q] = bitval;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < row_elems; e += blockDim.x) {
    pmask[e] = qmask[e % B];
    pbitval[e] = qbitval[e % B];
  }
}

// ---------------------------------------------------------------- compress
struct PosCompressArgs {
  const uint8_t *rows;
  int64_t n_rows;
  uint8_t *slots;
  int64_t slot_bytes;
  uint32_t *bitmask;
  uint32_t *row_bits;
  const uint32_t *pmask, *pbitval;
  Geo g;
  int64_t raw_bytes;
  int warps;
  int hdr_words;
  int warp_bytes;
  int table_bytes;
};

__device__ __forceinline__ void pos_prefetch(const PosCompressArgs &a, int64_t r, uint32_t *RAW) {
  if (r < a.n_rows) {
    const uint8_t *src = a.rows + r * a.raw_bytes;
    const int nvec = a.g.raw_words / 4;
    for (int v = threadIdx.x & 31; v < nvec; v += 32)
      cp_async16(reinterpret_cast<uint8_t *>(RAW) + 16 * v, src + 16 * v);
  }
  cp_async_commit();
}

template <int LWB>
__device__ bool pos_compress_row(const PosCompressArgs &a, const Tables &t, int64_t r,
                                 const uint32_t *RAW, uint32_t *OUT, uint32_t *HDR) {
  constexpr int GS = LWB / 4;   // lanes per block
  constexpr int BPS = 32 / GS;  // blocks per 128-word span
  const Geo &g = a.g;
  const int lane = threadIdx.x & 31;
  const int nvec = g.raw_words / 4;
  const int nspan = (g.raw_words + 127) >> 7;
  const uint4 *RAW4 = reinterpret_cast<const uint4 *>(RAW);

  // participation bits: a lane's four lane words against their own masks, a block's
  // bit the AND of its lanes' votes (lanes past the row vote "match")
  uint32_t hacc = 0;
  for (int i = 0; i < nspan; ++i) {
    const int v = 32 * i + lane;
    bool ok = true;
    if (v < nvec) {
      const uint4 x = RAW4[v];
      const int k = 4 * v;
      ok = ((x.x & t.M[k]) == t.V[k]) & ((x.y & t.M[k + 1]) == t.V[k + 1]) &
           ((x.z & t.M[k + 2]) == t.V[k + 2]) & ((x.w & t.M[k + 3]) == t.V[k + 3]);
    }
    uint32_t A = __ballot_sync(FULL, ok);
#pragma unroll
    for (int sft = 1; sft < GS; sft <<= 1) A &= A >> sft;
    uint32_t frag = 0;
#pragma unroll
    for (int j = 0; j < BPS; ++j) frag |= ((A >> (GS * j)) & 1u) << j;
    const int b0 = i * BPS;
    if (b0 + BPS > g.nb) frag &= low_mask((uint32_t)(g.nb - b0));
    hacc |= frag << (b0 & 31);
    if (((b0 + BPS) & 31) == 0 || b0 + BPS >= g.nb) {
      if (lane == 0) HDR[b0 >> 5] = hacc;
      hacc = 0;
    }
  }
  __syncwarp();
  // row bits: nb + sum over blocks of FB (matching) or 32 * lane words (raw)
  uint32_t part = 0;
  for (int b = lane; b < g.nb; b += 32) {
    const bool p = (HDR[b >> 5] >> (b & 31)) & 1u;
    part += p ? t.FB[b] : 32u * block_words(g, b);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(FULL, part, o);
  const uint32_t total = (uint32_t)g.nb + part;
  const uint32_t sw = (total + 31) >> 5;
  const bool comp = (int64_t)sw * 4 < a.raw_bytes;
  if (a.row_bits && lane == 0) a.row_bits[r] = total;

  uint4 *dst = reinterpret_cast<uint4 *>(a.slots + r * a.slot_bytes);
  if (!comp) {
    for (int v = lane; v < nvec; v += 32) dst[v] = RAW4[v];
    return false;
  }
  const uint32_t nout = (sw + 3) & ~3u;
  for (uint32_t v = lane; v < nout / 4; v += 32)
    reinterpret_cast<uint4 *>(OUT)[v] = make_uint4(0u, 0u, 0u, 0u);
  __syncwarp();
  const uint32_t nhw = ((uint32_t)g.nb + 31) >> 5;
  for (uint32_t q = lane; q < nhw; q += 32) OUT[q] = HDR[q];
  __syncwarp();
  uint32_t base = (uint32_t)g.nb;
  for (int i = 0; i < nspan; ++i) {
    const int v = 32 * i + lane;
    const bool in = v < nvec;
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (in) x = RAW4[v];
    const int k = 4 * v;
    const uint32_t blk = (uint32_t)k / LWB;
    const bool p = in && ((HDR[blk >> 5] >> (blk & 31)) & 1u);
    uint32_t c0, c1, c2, c3, T;
    if (!p) {
      c0 = x.x;
      c1 = x.y;
      c2 = x.z;
      c3 = x.w;
      T = in ? 128u : 0u;
    } else {
      const uint32_t F0 = t.F[k], F1 = t.F[k + 1], F2 = t.F[k + 2], F3 = t.F[k + 3];
      const uint64_t f0 = extract_runs(x.x, ~t.M[k]), f1 = extract_runs(x.y, ~t.M[k + 1]);
      const uint64_t f2 = extract_runs(x.z, ~t.M[k + 2]), f3 = extract_runs(x.w, ~t.M[k + 3]);
      const uint64_t lo = f0 | (f1 << F0), hi = f2 | (f3 << F2);  // F0 + F1 <= 64 bits each
      const uint32_t L01 = F0 + F1;
      uint64_t w01, w23;
      if (L01 == 0) {
        w01 = hi;
        w23 = 0;
      } else if (L01 == 64) {
        w01 = lo;
        w23 = hi;
      } else {
        w01 = lo | (hi << L01);
        w23 = hi >> (64 - L01);
      }
      c0 = (uint32_t)w01;
      c1 = (uint32_t)(w01 >> 32);
      c2 = (uint32_t)w23;
      c3 = (uint32_t)(w23 >> 32);
      T = L01 + F2 + F3;
    }
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
      const uint32_t nw = (sh + T + 31) >> 5;  // words touched (1..5)
      atomicOr(&OUT[q], c0 << sh);
      if (nw > 1) atomicOr(&OUT[q + 1], __funnelshift_l(c0, c1, sh));
      if (nw > 2) atomicOr(&OUT[q + 2], __funnelshift_l(c1, c2, sh));
      if (nw > 3) atomicOr(&OUT[q + 3], __funnelshift_l(c2, c3, sh));
      if (nw > 4) atomicOr(&OUT[q + 4], __funnelshift_l(c3, 0u, sh));
    }
  }
  __syncwarp();
  for (uint32_t v = lane; v < nout / 4; v += 32) dst[v] = reinterpret_cast<const uint4 *>(OUT)[v];
  return true;
}

template <int LWB>
__global__ void __launch_bounds__(POS_THREADS) pos_compress_kernel(PosCompressArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const Tables t = carve_tables(smem, a.g);
  build_tables(a.pmask, a.pbitval, a.g, t);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  if (warp >= a.warps) return;
  uint8_t *mine = smem + a.table_bytes + (size_t)warp * a.warp_bytes;
  uint32_t *HDR = reinterpret_cast<uint32_t *>(mine);
  uint32_t *RAW0 = HDR + a.hdr_words;
  uint32_t *OUT = RAW0 + 2 * a.g.raw_words;
  const int64_t first = (int64_t)blockIdx.x * a.warps + warp;
  const int64_t step = (int64_t)gridDim.x * a.warps;
  if (first == 0 && lane == 0 && (a.n_rows & 31))
    atomicAnd(&a.bitmask[a.n_rows >> 5], low_mask((uint32_t)(a.n_rows & 31)));
  if (first >= a.n_rows) return;
  pos_prefetch(a, first, RAW0);
  int b = 0;
  for (int64_t r = first; r < a.n_rows; r += step) {
    pos_prefetch(a, r + step, RAW0 + (b ^ 1) * a.g.raw_words);  // no-op past the end
    cp_async_wait<1>();
    __syncwarp();
    const bool comp = pos_compress_row<LWB>(a, t, r, RAW0 + b * a.g.raw_words, OUT, HDR);
    if (lane == 0) {
      const uint32_t bit = 1u << (r & 31);
      if (comp) atomicOr(&a.bitmask[r >> 5], bit);
      else atomicAnd(&a.bitmask[r >> 5], ~bit);
    }
    __syncwarp();
    b ^= 1;
  }
  cp_async_wait<0>();
}

// ---------------------------------------------------------------- gather
struct PosGatherArgs {
  const uint8_t *slots;
  int64_t slot_bytes;
  int64_t n_rows;
  const uint32_t *bitmask;
  const uint32_t *pmask, *pbitval;
  const int64_t *idx;
  int64_t n_idx;
  uint32_t *out;
  int32_t *status;
  Geo g;
  int64_t raw_bytes;
  int warps;
  int buf_bytes;   // one staging buffer: the raw row + 16 bytes
  int boff_words;  // per-warp block offsets
  int table_bytes;
};

// Stage the raw-size prefix of row r's slot (nothing for a bad index).
__device__ __forceinline__ void pos_stage(const PosGatherArgs &a, int64_t r, uint8_t *buf) {
  if (r >= 0 && r < a.n_rows) {
    const uint8_t *src = a.slots + r * a.slot_bytes;
    const int nvec = a.g.raw_words / 4;
    for (int v = threadIdx.x & 31; v < nvec; v += 32) cp_async16(buf + 16 * v, src + 16 * v);
  }
  cp_async_commit();
}

__device__ void pos_decode(const PosGatherArgs &a, const Tables &t, int64_t i, int64_t r,
                           const uint8_t *buf, uint32_t *BOFF) {
  const Geo &g = a.g;
  const int lane = threadIdx.x & 31;
  if (r < 0 || r >= a.n_rows) {
    if (lane == 0) report(a.status, IBP_ERR_INDEX);
    return;
  }
  const int nvec = g.raw_words / 4;
  uint4 *dst = reinterpret_cast<uint4 *>(a.out + i * (int64_t)g.raw_words);
  const uint32_t *S = reinterpret_cast<const uint32_t *>(buf);
  if (!((__ldg(a.bitmask + (r >> 5)) >> (r & 31)) & 1u)) {  // stored raw
    const uint4 *S4 = reinterpret_cast<const uint4 *>(buf);
    for (int v = lane; v < nvec; v += 32) dst[v] = S4[v];
    return;
  }
  // block offsets: exclusive warp scan of block sizes, 32 blocks per round
  uint32_t carry = (uint32_t)g.nb;
  for (int b0 = 0; b0 < g.nb; b0 += 32) {
    const int b = b0 + lane;
    uint32_t sz = 0;
    if (b < g.nb) sz = ((S[b >> 5] >> (b & 31)) & 1u) ? t.FB[b] : 32u * block_words(g, b);
    uint32_t incl = sz;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += y;
    }
    if (b < g.nb) BOFF[b] = carry + incl - sz;
    carry += __shfl_sync(FULL, incl, 31);
  }
  // carry = the row's bits; a stream of at least the raw size was never stored
  if ((int64_t)((carry + 31) >> 5) * 4 >= a.raw_bytes) {
    if (lane == 0) report(a.status, IBP_ERR_CORRUPT);
    return;
  }
  __syncwarp();
  for (int v = lane; v < nvec; v += 32) {
    uint32_t y[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = 4 * v + j;
      const int b = k >> g.lwb_shift;
      const bool p = (S[b >> 5] >> (b & 31)) & 1u;
      const uint32_t pos = BOFF[b] + (p ? (uint32_t)t.OFF[k] : 32u * (uint32_t)(k - b * g.lwb));
      const uint32_t wv = window(S[pos >> 5], S[(pos >> 5) + 1], pos & 31u);
      y[j] = p ? (deposit_runs(wv & low_mask(t.F[k]), ~t.M[k]) | t.V[k]) : wv;
    }
    dst[v] = make_uint4(y[0], y[1], y[2], y[3]);
  }
}

__global__ void __launch_bounds__(POS_THREADS) pos_gather_kernel(PosGatherArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const Tables t = carve_tables(smem, a.g);
  build_tables(a.pmask, a.pbitval, a.g, t);
  const int warp = threadIdx.x >> 5;
  if (warp >= a.warps) return;
  uint8_t *mine = smem + a.table_bytes +
                  (size_t)warp * (2 * (size_t)a.buf_bytes + 4 * (size_t)a.boff_words);
  uint8_t *buf0 = mine;
  uint32_t *BOFF = reinterpret_cast<uint32_t *>(mine + 2 * (size_t)a.buf_bytes);
  const int64_t step = (int64_t)gridDim.x * a.warps;
  int64_t i = (int64_t)blockIdx.x * a.warps + warp;
  if (i >= a.n_idx) return;
  int64_t r = __ldg(a.idx + i);
  pos_stage(a, r, buf0);
  int b = 0;
  for (; i < a.n_idx; i += step) {
    const int64_t i_next = i + step;
    const int64_t r_next = i_next < a.n_idx ? __ldg(a.idx + i_next) : -1;
    pos_stage(a, r_next, buf0 + (b ^ 1) * a.buf_bytes);  // nothing past the end
    cp_async_wait<1>();
    __syncwarp();
    pos_decode(a, t, i, r, buf0 + b * a.buf_bytes, BOFF);
    __syncwarp();
    r = r_next;
    b ^= 1;
  }
  cp_async_wait<0>();
}

template <typename K>
int one_wave_grid(K kernel, size_t smem, int64_t want, const DeviceInfo &dev, int *grid) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, POS_THREADS, smem) !=
          cudaSuccess ||
      per_sm < 1)
    return IBP_ERR_CUDA;
  *grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)dev.sm_count * per_sm));
  return IBP_OK;
}

int ilog2i(int x) {
  int s = 0;
  while ((1 << s) < x) ++s;
  return s;
}

Geo geo_of(const RowGeom &g) {
  Geo o;
  o.w = g.w;
  o.lwb = g.lwb;
  o.lwb_shift = ilog2i(g.lwb);
  o.lwt = g.lwt;
  o.nb = g.nb;
  o.raw_words = g.raw_words;
  return o;
}

template <int LWB>
int launch_pos_compress(const PosCompressArgs &a, size_t smem, int64_t n_rows,
                        const DeviceInfo &dev, cudaStream_t s) {
  if (cudaFuncSetAttribute(pos_compress_kernel<LWB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return IBP_ERR_CUDA;
  int grid = 0;
  if (int rc = one_wave_grid(pos_compress_kernel<LWB>, smem, (n_rows + a.warps - 1) / a.warps,
                             dev, &grid))
    return rc;
  pos_compress_kernel<LWB><<<grid, POS_THREADS, smem, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

}  // namespace

size_t pos_scratch_bytes(const RowGeom &g) { return (size_t)g.raw_words * 32 * 8; }

int launch_build_meta_positions(const void *rows, int64_t n_rows, const RowGeom &g, double T,
                                uint32_t *d_pmask, uint32_t *d_pbitval, void *d_scratch,
                                cudaStream_t s, bool per_block_position) {
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  unsigned long long *counters = static_cast<unsigned long long *>(d_scratch);
  if (cudaMemsetAsync(counters, 0, pos_scratch_bytes(g), s) != cudaSuccess) return IBP_ERR_CUDA;
  // about two resident threads' worth of work per SM slot, every column covered
  const int64_t target = (int64_t)dev.sm_count * 2048;
  const int64_t n_chunks = std::max<int64_t>(1, std::min<int64_t>(n_rows, target / g.raw_words));
  const int64_t rows_per_chunk = (n_rows + n_chunks - 1) / n_chunks;
  const int64_t threads = (int64_t)g.raw_words * n_chunks;
  const int64_t blocks = (threads + POS_THREADS - 1) / POS_THREADS;
  pos_count_kernel<<<(unsigned)blocks, POS_THREADS, 0, s>>>(
      static_cast<const uint32_t *>(rows), n_rows, g.raw_words, rows_per_chunk, n_chunks,
      counters);
  if (cudaGetLastError() != cudaSuccess) return IBP_ERR_CUDA;
  if (per_block_position)
    pos_block_finalize_kernel<<<1, 256, 0, s>>>(counters, n_rows, (int)g.row_elems, g.w, g.B, T,
                                                d_pmask, d_pbitval);
  else
    pos_finalize_kernel<<<(unsigned)((g.row_elems + 127) / 128), 128, 0, s>>>(
        counters, n_rows, (int)g.row_elems, g.w, T, d_pmask, d_pbitval);
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

int launch_compress_positions(const void *rows, int64_t n_rows, const RowGeom &g,
                              const uint32_t *d_pmask, const uint32_t *d_pbitval, void *slots,
                              int64_t slot_bytes, uint32_t *d_bitmask, uint32_t *d_row_bits,
                              cudaStream_t s) {
  if (n_rows == 0) return IBP_OK;
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  PosCompressArgs a;
  a.rows = static_cast<const uint8_t *>(rows);
  a.n_rows = n_rows;
  a.slots = static_cast<uint8_t *>(slots);
  a.slot_bytes = slot_bytes;
  a.bitmask = d_bitmask;
  a.row_bits = d_row_bits;
  a.pmask = d_pmask;
  a.pbitval = d_pbitval;
  a.g = geo_of(g);
  a.raw_bytes = g.raw_bytes;
  a.hdr_words = (((g.nb + 31) / 32) + 3) & ~3;
  a.warp_bytes = 4 * (a.hdr_words + 3 * g.raw_words);  // header, two staged rows, stream
  a.table_bytes = (int)table_bytes(g.raw_words, g.nb);
  const int budget = std::min(POS_SMEM_BUDGET, dev.max_smem_optin - 1024) - a.table_bytes;
  a.warps = std::min(POS_WARPS, budget / a.warp_bytes);
  if (a.warps < 1) return IBP_ERR_UNSUPPORTED;
  const size_t smem = (size_t)a.table_bytes + (size_t)a.warps * a.warp_bytes;
  switch (g.lwb) {
    case 8: return launch_pos_compress<8>(a, smem, n_rows, dev, s);
    case 16: return launch_pos_compress<16>(a, smem, n_rows, dev, s);
    case 32: return launch_pos_compress<32>(a, smem, n_rows, dev, s);
    default: return launch_pos_compress<64>(a, smem, n_rows, dev, s);
  }
}

int launch_gather_positions(const void *slots, int64_t slot_bytes, int64_t n_rows,
                            const RowGeom &g, const uint32_t *d_bitmask, const uint32_t *d_pmask,
                            const uint32_t *d_pbitval, const int64_t *d_idx, int64_t n_idx,
                            void *out, int32_t *d_status, cudaStream_t s) {
  if (n_idx == 0) return IBP_OK;
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  PosGatherArgs a;
  a.slots = static_cast<const uint8_t *>(slots);
  a.slot_bytes = slot_bytes;
  a.n_rows = n_rows;
  a.bitmask = d_bitmask;
  a.pmask = d_pmask;
  a.pbitval = d_pbitval;
  a.idx = d_idx;
  a.n_idx = n_idx;
  a.out = static_cast<uint32_t *>(out);
  a.status = d_status;
  a.g = geo_of(g);
  a.raw_bytes = g.raw_bytes;
  a.buf_bytes = (int)align16((size_t)g.raw_bytes + 16);
  a.boff_words = (int)((g.nb + 3) & ~3);
  a.table_bytes = (int)table_bytes(g.raw_words, g.nb);
  const int per_warp = 2 * a.buf_bytes + 4 * a.boff_words;
  const int budget = std::min(POS_SMEM_BUDGET, dev.max_smem_optin - 1024) - a.table_bytes;
  a.warps = std::min(POS_WARPS, budget / per_warp);
  if (a.warps < 1) return IBP_ERR_UNSUPPORTED;
  const size_t smem = (size_t)a.table_bytes + (size_t)a.warps * per_warp;
  if (cudaFuncSetAttribute(pos_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return IBP_ERR_CUDA;
  int grid = 0;
  if (int rc = one_wave_grid(pos_gather_kernel, smem, (n_idx + a.warps - 1) / a.warps, dev, &grid))
    return rc;
  pos_gather_kernel<<<grid, POS_THREADS, smem, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

}  // namespace ibp
