// Saving-aware metadata for Invariant Bit Packing on sm_103a.
//
// "Reducing the GPU Memory Bottleneck with Lossless Compression for ML --
// Extended", technical summary, "Core algorithm": preprocessing keeps every bit
// position whose value is shared by a fraction T of the sample, and compression
// strips a block's invariant bits only when all of them hold in all of its
// elements. A position kept by the threshold rule whose rare exceptions are spread
// over many blocks can therefore cost more blocks than it saves bits. This variant
// scores a nested family of masks on the data and keeps the cheapest one:
//   candidate 0 = the threshold mask M0; candidate k+1 = candidate k minus its
//   least-held positions (equal majority counts leave together); last = empty.
//
// Four launches on one stream:
//   1. the positional population count of the preprocessing stage (shared);
//   2. select_groups_kernel (one warp): M0, bitval, and the candidate masks;
//   3. select_score_kernel: one pass over the rows. A warp owns a contiguous range
//      of rows and walks them in 128-word chunks (a 16-byte load per lane, four
//      chunks in flight). For each block it ORs the mismatch bits
//      (x ^ bitval) & M0 over the block's words and finds the block's level: the
//      first candidate whose mask misses all of them (byte-table lookups of the
//      largest group rank among the bits). Lane k then counts, per row, the blocks
//      whose level is <= k,
//      i.e. the blocks that match candidate k, turns that into the row's stored
//      bytes under candidate k, and accumulates them; one 64-bit atomic per lane
//      and warp at the end;
//   4. select_finalize_kernel (one warp): the lowest score wins (ties: lower k),
//      written as an ibp_meta, plus the optional candidate table.
// The empty mask never compresses a row (nb*(1 + B*w) bits > the raw row), so a
// 33rd candidate (all 32 positions in M0 with 32 distinct counts) is scored as
// n_rows raw rows without a lane of its own.
#include <algorithm>
#include <atomic>
#include <climits>

#include "ibp_device.cuh"
#include "ibp_internal.h"

namespace ibp {
namespace {

constexpr int SEL_THREADS = 256;
constexpr int SEL_WARPS = SEL_THREADS / 32;
constexpr int NCAND = IBP_MAX_MASK_CANDIDATES;  // w + 1 at most
constexpr int SEL_UNROLL = 4;                   // chunks in flight per warp

struct SelectScratch {
  unsigned long long counters[32];  // ones per bit position of the 32-bit words
  unsigned long long score[32];     // bytes of the rows under candidate k (k < 32)
  uint32_t keep[NCAND];             // candidate masks (w bits), 0 past the last
  uint32_t n_cand;                  // number of candidates (1 .. w+1)
  uint32_t bitval0;                 // bitval of M0
  uint8_t level[32];                // position j: 1 + its group rank if in M0, else 0
};

__global__ void select_groups_kernel(SelectScratch *sc, int64_t n_elems, int w, double T) {
  const int j = threadIdx.x;  // one warp; lane j = bit position j
  unsigned long long c1 = 0;  // element bit j: bits j, j + w, ... of the 32-bit words
  if (j < w)
    for (int q = j; q < 32; q += w) c1 += sc->counters[q];
  const unsigned long long N = (unsigned long long)n_elems;
  const unsigned long long c0 = N - c1;
  const bool v = c1 > c0;  // a tie keeps 0
  const unsigned long long held = v ? c1 : c0;
  const bool inv = j < w && (double)held >= T * (double)N;
  const uint32_t mask0 = __ballot_sync(FULL, inv);
  const uint32_t bitval0 = __ballot_sync(FULL, inv && v);
  // lane j is the first invariant position holding its count?
  bool first = inv;
  for (int i = 0; i < 32; ++i) {
    const unsigned long long hi = __shfl_sync(FULL, held, i);
    if (i < j && ((mask0 >> i) & 1u) && hi == held) first = false;
  }
  const uint32_t reps = __ballot_sync(FULL, first);
  // group rank: how many distinct counts among M0's positions are below this one
  int rank = 0;
  for (int i = 0; i < 32; ++i) {
    const unsigned long long hi = __shfl_sync(FULL, held, i);
    if (((reps >> i) & 1u) && hi < held) ++rank;
  }
  const int groups = __popc(reps);
  for (int k = 0; k < NCAND; ++k) {
    const uint32_t mk = __ballot_sync(FULL, inv && rank >= k);
    if (j == 0) sc->keep[k] = (k <= groups) ? mk : 0u;
  }
  // a block whose mismatch bits include position j matches candidate k iff k > rank
  sc->level[j] = inv ? (uint8_t)(rank + 1) : (uint8_t)0;
  if (j == 0) {
    sc->n_cand = (uint32_t)groups + 1;
    sc->bitval0 = bitval0;
  }
}

struct ScoreArgs {
  const uint4 *rows;
  int64_t n_rows;
  int vpr;  // 16-byte vectors per row (raw_words / 4)
  int nb;
  int B;
  int bt;   // elements of the last block (B, or fewer for a shorter tail)
  int w;
  int64_t raw_bytes;
  SelectScratch *sc;
};

// LWB = 32-bit words per block (8, 16, 32 or 64): a block spans LWB/4 lanes of a
// 128-word chunk, and a chunk holds 32/(LWB/4) whole blocks. A shorter last block
// spans fewer lanes; the lanes past the row's end load bitval, which adds no
// mismatch bit, so the OR over the block's lane group is the last block's own.
//
// A block's level is the largest level[j] over its mismatch bits j (0 if none):
// the block matches candidate k iff k >= level. It is read from four 256-entry
// byte tables (one per byte of the lane word: the largest level among the byte's
// set bits), so a block costs four shared-memory lookups.
template <int LWB>
__global__ void __launch_bounds__(SEL_THREADS) select_score_kernel(const ScoreArgs a) {
  constexpr int LPB = LWB / 4;
  constexpr int BPC = 32 / LPB;
  __shared__ uint8_t lvl_tab[4][256];
  __shared__ uint32_t s_M0, s_bv2, s_keep[32];
  {
    const int b = threadIdx.x >> 6;  // 256 threads: 4 tables x 64 threads x 4 entries
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int x = ((threadIdx.x & 63) << 2) + q;
      int mx = 0;
      for (int i = 0; i < 8; ++i)
        if ((x >> i) & 1) {
          const int pos = (8 * b + i) & (a.w - 1);  // 16-bit words: both halves alike
          mx = max(mx, (int)a.sc->level[pos]);
        }
      lvl_tab[b][x] = (uint8_t)mx;
    }
  }
  if (threadIdx.x < 32) s_keep[threadIdx.x] = a.sc->keep[threadIdx.x];
  if (threadIdx.x == 0) {
    s_M0 = replicate(a.sc->keep[0], a.w);
    s_bv2 = replicate(a.sc->bitval0, a.w);
  }
  __syncthreads();
  const uint32_t M0 = s_M0, bv2 = s_bv2;
  const int lane = threadIdx.x & 31;
  const uint32_t wmask = low_mask((uint32_t)a.w);
  // field width under candidate `lane`; bits of a matching / a raw full block, and
  // of the last block matching / raw
  const uint32_t mk = (uint32_t)(a.w - __popc(s_keep[lane] & wmask));
  const uint32_t bm = (uint32_t)a.B * mk;
  const uint32_t br = (uint32_t)a.B * (uint32_t)a.w;
  const uint32_t tm = (uint32_t)a.bt * mk;
  const uint32_t tr = (uint32_t)a.bt * (uint32_t)a.w;
  const uint32_t raw = (uint32_t)a.raw_bytes;
  const uint32_t nb = (uint32_t)a.nb;
  const int cpr = (a.vpr + 31) / 32;  // chunks per row

  const int64_t warps = (int64_t)gridDim.x * SEL_WARPS;
  const int64_t wid = (int64_t)blockIdx.x * SEL_WARPS + threadIdx.x / 32;
  const int64_t per = (a.n_rows + warps - 1) / warps;
  int64_t r = wid * per;
  const int64_t r_end = min(a.n_rows, r + per);
  int c = 0;
  uint32_t matched = 0;    // full blocks of the row matching candidate `lane`
  bool tail_match = false;  // the row's last block matches it
  unsigned long long acc = 0;
  while (r < r_end) {
    uint4 x[SEL_UNROLL];
    int cc[SEL_UNROLL];
    bool ok[SEL_UNROLL];
    int64_t pr = r;
    int pc = c;
#pragma unroll
    for (int u = 0; u < SEL_UNROLL; ++u) {
      ok[u] = pr < r_end;
      cc[u] = pc;
      const int vec = pc * 32 + lane;
      x[u] = (ok[u] && vec < a.vpr) ? a.rows[pr * a.vpr + vec] : make_uint4(bv2, bv2, bv2, bv2);
      if (++pc == cpr) {
        pc = 0;
        ++pr;
      }
    }
#pragma unroll
    for (int u = 0; u < SEL_UNROLL; ++u) {
      if (!ok[u]) break;  // warp-uniform
      uint32_t D = ((x[u].x ^ bv2) | (x[u].y ^ bv2) | (x[u].z ^ bv2) | (x[u].w ^ bv2)) & M0;
#pragma unroll
      for (int o = 1; o < LPB; o <<= 1) D |= __shfl_xor_sync(FULL, D, o);
      const int lv = max(max((int)lvl_tab[0][D & 0xFFu], (int)lvl_tab[1][(D >> 8) & 0xFFu]),
                         max((int)lvl_tab[2][(D >> 16) & 0xFFu], (int)lvl_tab[3][D >> 24]));
      const uint32_t blk0 = (uint32_t)(cc[u] * BPC);
#pragma unroll
      for (int b = 0; b < BPC; ++b) {
        const int lb = __shfl_sync(FULL, lv, b * LPB);
        const uint32_t blk = blk0 + b;
        if (blk + 1 < nb) matched += (lb <= lane) ? 1u : 0u;
        else if (blk + 1 == nb) tail_match = lb <= lane;
      }
      if (cc[u] == cpr - 1) {  // the row is complete
        const uint32_t bits = nb + matched * bm + (nb - 1 - matched) * br + (tail_match ? tm : tr);
        const uint32_t stored = ((bits + 31u) >> 5) << 2;
        acc += stored < raw ? stored : raw;
        matched = 0;
      }
    }
    r = pr;
    c = pc;
  }
  if (acc) atomicAdd(&a.sc->score[lane], acc);
}

__global__ void select_finalize_kernel(const SelectScratch *sc, int64_t n_rows, int64_t raw_bytes,
                                       uint32_t dtype, uint32_t block_elems, ibp_meta *meta,
                                       ibp_mask_candidate *cand) {
  const int k = threadIdx.x;  // one warp; lane k = candidate k
  const int n_cand = (int)sc->n_cand;
  const long long all_raw = (long long)(n_rows * raw_bytes);
  const long long score = (k < n_cand) ? (long long)sc->score[k] : -1;
  // lowest score, ties to the lower k; candidate 32 (the empty mask) scores all_raw,
  // the highest possible score, so it never beats a lower k
  long long best = (k < n_cand) ? score : LLONG_MAX;
  int best_k = (k < n_cand) ? k : NCAND;
  for (int o = 16; o > 0; o >>= 1) {
    const long long ob = __shfl_xor_sync(FULL, best, o);
    const int ok = __shfl_xor_sync(FULL, best_k, o);
    if (ob < best || (ob == best && ok < best_k)) {
      best = ob;
      best_k = ok;
    }
  }
  const uint32_t bitval0 = sc->bitval0;
  if (k == 0) {
    ibp_meta m;
    m.mask = sc->keep[best_k];
    m.bitval = bitval0 & m.mask;
    m.dtype = dtype;
    m.block_elems = block_elems;
    *meta = m;
  }
  if (cand) {
    ibp_mask_candidate e;
    e.mask = (k < n_cand) ? sc->keep[k] : 0u;
    e.bitval = bitval0 & e.mask;
    e.stored_bytes = score;
    cand[k] = e;
    if (k == 0) {
      ibp_mask_candidate last;
      last.mask = 0u;
      last.bitval = 0u;
      last.stored_bytes = (n_cand == NCAND) ? all_raw : -1;
      cand[NCAND - 1] = last;
    }
  }
}

// One wave of resident CTAs: every warp gets an equal share of rows, so a second
// partial wave would only lengthen the tail.
template <int LWB>
int launch_score(const ScoreArgs &a, const DeviceInfo &dev, cudaStream_t s) {
  static std::atomic<int> occupancy{0};  // resident CTAs per SM, looked up once
  int per_sm = occupancy.load(std::memory_order_relaxed);
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, select_score_kernel<LWB>, SEL_THREADS,
                                                      0) != cudaSuccess || n < 1)
      n = 1;
    per_sm = n;
    occupancy.store(n, std::memory_order_relaxed);
  }
  const int64_t want = std::max<int64_t>(1, (a.n_rows + SEL_WARPS - 1) / SEL_WARPS);
  const int grid = (int)std::min<int64_t>(want, (int64_t)dev.sm_count * per_sm);
  select_score_kernel<LWB><<<grid, SEL_THREADS, 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

}  // namespace

size_t select_scratch_bytes() { return 1024; }
static_assert(sizeof(SelectScratch) <= 1024, "select scratch layout outgrew its size");

int launch_build_meta_select(const void *rows, int64_t n_rows, const RowGeom &g, uint32_t dtype,
                             double T, ibp_meta *d_meta, ibp_mask_candidate *d_candidates,
                             void *d_scratch, cudaStream_t s) {
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  SelectScratch *sc = static_cast<SelectScratch *>(d_scratch);
  if (cudaMemsetAsync(sc, 0, sizeof(SelectScratch), s) != cudaSuccess) return IBP_ERR_CUDA;
  const int64_t n_elems = n_rows * g.row_elems;
  if (int rc = launch_meta_count(rows, n_elems * g.w / 32, sc->counters, s)) return rc;
  select_groups_kernel<<<1, 32, 0, s>>>(sc, n_elems, g.w, T);
  if (cudaGetLastError() != cudaSuccess) return IBP_ERR_CUDA;
  ScoreArgs a;
  a.rows = static_cast<const uint4 *>(rows);
  a.n_rows = n_rows;
  a.vpr = g.raw_words / 4;
  a.nb = g.nb;
  a.B = g.B;
  a.bt = g.lwt * 32 / g.w;
  a.w = g.w;
  a.raw_bytes = g.raw_bytes;
  a.sc = sc;
  int rc;
  switch (g.lwb) {
    case 8: rc = launch_score<8>(a, dev, s); break;
    case 16: rc = launch_score<16>(a, dev, s); break;
    case 32: rc = launch_score<32>(a, dev, s); break;
    case 64: rc = launch_score<64>(a, dev, s); break;
    default: return IBP_ERR_UNSUPPORTED;
  }
  if (rc) return rc;
  select_finalize_kernel<<<1, 32, 0, s>>>(sc, n_rows, g.raw_bytes, dtype, (uint32_t)g.B, d_meta,
                                          d_candidates);
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

}  // namespace ibp
