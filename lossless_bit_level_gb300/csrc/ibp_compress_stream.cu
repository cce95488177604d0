// Compression of long rows (over 2 KiB, up to the longest row the library accepts)
// for sm_103a: one warp per row, one pass over the row, no CTA barriers.
//
// "Reducing the GPU Memory Bottleneck with Lossless Compression for ML --
// Extended", technical summary, "Core algorithm" (compression: per-block match
// test, participation bit, invariant bits stripped, remaining bits packed) and
// "System integration" (fixed-size slot per row, GPU bitmask). Same stream as the
// other compression kernels.
//
// Every block is B*m bits when it matches and B*w bits when it does not, and B is
// 32 or 64, so both are whole 32-bit words: past the nb participation bits, each
// block starts on a word boundary of the "payload" (the stream without its first nb
// bits). Stream word q >= nb/32 is payload word q - nb/32 moved up by nb mod 32 bits
// over the top of the payload word before it.
//
// A warp walks its row in steps of 512 bytes (128 lane words), staged with cp.async
// PF - 1 steps ahead (lane l copies the 16-byte vector 32k + l of step k). Per step:
//   * match bits: per 32 lane words a vote of "my lane word matches", combined per
//     block, into the row's participation bits (kept per warp in shared memory and
//     written into the slot when the row ends);
//   * while no block of the row has matched yet, the row can only end up stored
//     raw (its stream is nb bits longer than the row), so the vectors are copied to
//     the slot as they are: rows that never match are read once and written once. At
//     the first matching block the row starts over from its first step in stream
//     mode;
//   * stream mode, 32 lane words at a time, one per lane: a raw block's payload words
//     are its lane words; a matching block's lane words give fields of fc bits, and
//     lane k assembles payload word k from the (at most three for fc >= 16) fields
//     that overlap it, fetched with shuffles (which fields, and the shifts, depend
//     only on k and fc). For fields of 8, 16 or 24 bits a full step is taken from
//     the 16-byte view instead (lane l holds lane words 4l..4l+3): its four fields
//     fill fc/8 whole payload words, which the lane writes itself, no shuffles. The
//     payload words go into a 256-word ring per warp, at the index of the stream word
//     they start;
//   * the complete 16-byte stream vectors (at most one per lane per step) go out to
//     the slot, each lane's words funnel-shifted from two payload words. The vectors that hold participation
//     bits are written last: those below the first payload word from the warp's copy
//     of the bits, the one shared with the payload (at most one) kept back from the
//     flush and written with the bits ORed in.
// The row's size is nb plus the payload bits; a row whose stream would not be
// shorter than the raw row is rewritten raw from the source (only rows that matched
// somewhere and still save nothing).
#include <algorithm>
#include <atomic>

#include "ibp_device.cuh"
#include "ibp_internal.h"

namespace ibp {
namespace {

// One warp per CTA, 24 CTAs per SM at 80 registers (measured on 22 KB rows: 49.8 us,
// against 52.9 with 2-warp CTAs and 56.0 with 8-warp CTAs at the same 24 warps per SM)
constexpr int SW_THREADS = 32;
constexpr int SW_WARPS = SW_THREADS / 32;
constexpr int SW_CTAS_PER_SM = 24;
constexpr int RING_WORDS = 256;   // payload words per warp; a step adds at most 128
constexpr int RING_VECS = RING_WORDS / 4;
constexpr int PF = 8;             // staging slots per warp: PF - 1 steps in flight

struct StreamArgs {
  const uint8_t *rows;
  int64_t n_rows;
  uint8_t *slots;
  int64_t slot_bytes;
  uint32_t *bitmask;
  uint32_t *row_bits;
  int32_t *status;
  const ibp_meta *meta;
  uint32_t dtype, block_elems;
  int nb, raw_words;
  int hdr_words;  // participation-bit words per warp: ceil(nb / 32) rounded up to 4
  int64_t raw_bytes;
};

// Per-warp shared memory (dynamic; every part 16-byte aligned): the staging slots, the
// payload ring, the one vector shared by participation bits and payload, then the
// row's participation bits (hdr_words words, a multiple of 4).
struct __align__(16) WarpFixed {
  uint4 stage[PF][32];  // the row's next steps, one 16-byte vector per lane (cp.async)
  uint32_t ring[RING_WORDS];
  uint4 head;
};

// The warp's part of shared memory: one base address, the parts at constant offsets.
struct WarpRing {
  uint8_t *base;
  __device__ __forceinline__ uint4 (*stage() const)[32] {
    return reinterpret_cast<WarpFixed *>(base)->stage;
  }
  __device__ __forceinline__ uint32_t *ring() const {
    return reinterpret_cast<WarpFixed *>(base)->ring;
  }
  __device__ __forceinline__ uint4 *head() const { return &reinterpret_cast<WarpFixed *>(base)->head; }
  __device__ __forceinline__ uint32_t *hdr() const {
    return reinterpret_cast<uint32_t *>(base + sizeof(WarpFixed));
  }
};

__host__ __device__ inline size_t warp_ring_bytes(int hdr_words) {
  return sizeof(WarpFixed) + 4 * (size_t)hdr_words;
}

__device__ __forceinline__ uint4 load_vec(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Per-lane constants of the packing of 32 (or SEG) fields of fc bits (fc > 0): payload
// word k (k = lane % SEG) starts in field i0 = 32k / fc, a0 bits into it; nt fields
// at most overlap one word; for fc >= 16 the three overlapping fields move up by l1
// and l2 bits (multipliers m1 = 2^l1, m2 = 2^l2; 0 when the field is not in the word).
struct PackLane {
  int i0;
  uint32_t a0;
  int nt;
  uint32_t l1, l2, m1, m2;
};

// Runs of kept bits, up to four, in registers (unused runs have an empty mask); a mask
// with more runs reads the run table from shared memory.
struct Runs4 {
  uint32_t sh[4], msrc[4];
  uint32_t mul[4];  // 2^(32 - sh): x >> sh as the high word of x * mul (1 <= sh <= 31)
  bool wide;        // more than four runs
};

__device__ __forceinline__ Runs4 load_runs4(const SharedRuns &s) {
  Runs4 r;
  r.wide = s.n > 4;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const bool use = (uint32_t)k < s.n && !r.wide;
    r.sh[k] = use ? s.sh[k] : 0u;
    r.msrc[k] = use ? s.msrc[k] : 0u;
    r.mul[k] = (r.sh[k] >= 1u && r.sh[k] <= 31u) ? 1u << (32u - r.sh[k]) : 0u;
  }
  return r;
}

__device__ __forceinline__ uint32_t extract4(uint32_t x, const Runs4 &r, const SharedRuns &s) {
  if (r.wide) return extract<-1>(x, RegRuns<-1>{}, s);
  return ((x >> r.sh[0]) & r.msrc[0]) | ((x >> r.sh[1]) & r.msrc[1]) |
         ((x >> r.sh[2]) & r.msrc[2]) | ((x >> r.sh[3]) & r.msrc[3]);
}

// extract4 for a mask whose first run starts at bit 0 (every later run has sh >= 1):
// the shifts run as multiplies on the FMA pipe, leaving the ALU pipe one AND-OR per
// run.
__device__ __forceinline__ uint32_t extract4_mul(uint32_t x, const Runs4 &r) {
  return (x & r.msrc[0]) | (__umulhi(x, r.mul[1]) & r.msrc[1]) |
         (__umulhi(x, r.mul[2]) & r.msrc[2]) | (__umulhi(x, r.mul[3]) & r.msrc[3]);
}

// Payload word `lane % SEG` of a matching segment of SEG fields of fc bits (field i
// from lane i of the segment, at bit i*fc).
template <int SEG>
__device__ __forceinline__ uint32_t pack_word(uint32_t f, uint32_t fc, const PackLane &pl) {
  uint32_t c = __shfl_sync(FULL, f, pl.i0, SEG) >> pl.a0;
  uint32_t l = fc - pl.a0;
  for (int t = 1; t < pl.nt; ++t, l += fc) {
    const uint32_t h = __shfl_sync(FULL, f, pl.i0 + t, SEG);
    c |= __funnelshift_lc(0u, h, l);  // h << l, 0 once l >= 32
  }
  return c;
}

// pack_word for 32 fields with fc >= 16 (at most three per word), the upper two moved
// up by multiplies (disjoint bits: add = OR).
__device__ __forceinline__ uint32_t pack3(uint32_t f, const PackLane &pl) {
  const uint32_t c0 = __shfl_sync(FULL, f, pl.i0);
  const uint32_t c1 = __shfl_sync(FULL, f, pl.i0 + 1);
  const uint32_t c2 = __shfl_sync(FULL, f, pl.i0 + 2);
  return c2 * pl.m2 + (c1 * pl.m1 + (c0 >> pl.a0));
}

// Match bits of one step from its lane words, 32 at a time (xg[g]: lane word 32g +
// lane, 0 past the row): bit j = block j of the step matches. Uniform over the warp.
template <int LWB>
__device__ __forceinline__ uint32_t group_frag(const uint32_t (&xg)[4], int nw_step, int nblk,
                                               const Code &code) {
  constexpr int SEG = LWB < 32 ? LWB : 32;
  constexpr int SPG = 32 / SEG;  // segments (blocks, or half blocks) per group
  const int lane = threadIdx.x & 31;
  uint32_t segbits = 0;  // bit (g * SPG + s): segment s of group g matches
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const bool ok = 32 * g + lane >= nw_step || ((xg[g] ^ code.bitval32) & code.mask32) == 0u;
    if (SEG == 32) {
      segbits |= (uint32_t)__all_sync(FULL, ok) << g;
    } else {
      uint32_t A = __ballot_sync(FULL, ok);
#pragma unroll
      for (int sft = 1; sft < SEG; sft <<= 1) A &= A >> sft;
#pragma unroll
      for (int s2 = 0; s2 < SPG; ++s2) segbits |= ((A >> (s2 * SEG)) & 1u) << (g * SPG + s2);
    }
  }
  uint32_t frag = segbits;
  if (LWB == 64) {  // a block is two groups: both halves must match
    frag = (segbits & (segbits >> 1)) & 0x5u;
    frag = (frag & 1u) | ((frag >> 1) & 2u);
  }
  return frag & low_mask((uint32_t)nblk);
}

// Row state in stream mode.
struct StreamPos {
  uint32_t pb;  // payload bits placed (whole words except after the row's last block)
  int fv;       // next stream vector to write out
};

// A full step (128 lane words of the row) of blocks of 32 or 64 lane words. FAST
// (fc >= 16, at most four runs of kept bits, bit 0 kept): one warp-uniform choice
// per step (every block packed, every block raw, or mixed), no branch within it.
template <int LWB, bool FAST>
__device__ __forceinline__ void pack_full(const Code &code, const Runs4 &runs,
                                          const SharedRuns &sruns, WarpRing &w,
                                          const uint32_t (&xg)[4], uint32_t frag, StreamPos &sp,
                                          int qh, const PackLane &pl) {
  const int lane = threadIdx.x & 31;
  const uint32_t fc = (uint32_t)code.fc;
  uint32_t wq = (uint32_t)qh + (sp.pb >> 5) + (uint32_t)lane;  // this lane's stream word
  constexpr uint32_t ALL = (1u << (128 / LWB)) - 1u;
  if (FAST && frag == ALL) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint32_t c = pack3(extract4_mul(xg[g], runs), pl);
      if ((uint32_t)lane < fc) w.ring()[wq & (RING_WORDS - 1)] = c;
      wq += fc;
    }
  } else if (frag == 0u) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      w.ring()[wq & (RING_WORDS - 1)] = xg[g];
      wq += 32u;
    }
  } else {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const bool p = (frag >> (32 * g / LWB)) & 1u;
      uint32_t c = 0u;
      if (FAST) c = pack3(extract4_mul(xg[g], runs), pl);
      else if (fc != 0u) c = pack_word<32>(extract4(xg[g], runs, sruns), fc, pl);
      const uint32_t n = p ? fc : 32u;
      if ((uint32_t)lane < n) w.ring()[wq & (RING_WORDS - 1)] = p ? c : xg[g];
      wq += n;
    }
  }
  sp.pb = (wq - (uint32_t)lane - (uint32_t)qh) << 5;
}

// Match bits of a full step from the 16-byte view (lane l holds lane words 4l..4l+3):
// a block is LWB / 4 consecutive lanes, and matches when all of their words do.
template <int LWB>
__device__ __forceinline__ uint32_t vec_frag(const uint4 &v, const Code &code) {
  constexpr int LPB = LWB / 4;  // lanes per block
  constexpr int BPS = 128 / LWB;
  const uint32_t bv = code.bitval32, m = code.mask32;
  const bool ok = (((v.x ^ bv) & m) | ((v.y ^ bv) & m) | ((v.z ^ bv) & m) | ((v.w ^ bv) & m)) == 0u;
  uint32_t A = __ballot_sync(FULL, ok);
#pragma unroll
  for (int sft = 1; sft < LPB; sft <<= 1) A &= A >> sft;
  if (LPB == 8) return ((A & 0x01010101u) * 0x01020408u) >> 24;  // bits 0, 8, 16, 24
  uint32_t frag = 0;
#pragma unroll
  for (int b = 0; b < BPS; ++b) frag |= ((A >> (b * LPB)) & 1u) << b;
  return frag;
}

// A full step packed from the 16-byte view, for fields of FC = 8, 16 or 24 bits: four
// consecutive lane words give four fields that fill FC / 8 whole payload words, so
// each lane writes its own words (no shuffles). A raw block's lane writes its four
// lane words.
template <int LWB, int FC>
__device__ __forceinline__ void pack_vec(const Runs4 &runs, WarpRing &w, const uint4 &v,
                                         uint32_t frag, StreamPos &sp, int qh) {
  static_assert(FC == 8 || FC == 16 || FC == 24, "whole words per four fields");
  constexpr int LPB = LWB / 4;
  constexpr int BPS = 128 / LWB;
  constexpr uint32_t MW = (uint32_t)LWB * FC / 32;  // payload words of a matching block
  const int lane = threadIdx.x & 31;
  const uint32_t blk = (uint32_t)lane / LPB, pos = (uint32_t)lane % LPB;
  const uint32_t p = (frag >> blk) & 1u;
  const uint32_t nm = __popc(frag & low_mask(blk));  // matching blocks before this one
  uint32_t wq = (uint32_t)qh + (sp.pb >> 5) + nm * MW + (blk - nm) * (uint32_t)LWB;
  uint32_t *ring = w.ring();
  if (p) {
    const uint32_t f0 = extract4_mul(v.x, runs), f1 = extract4_mul(v.y, runs);
    const uint32_t f2 = extract4_mul(v.z, runs), f3 = extract4_mul(v.w, runs);
    wq += pos * (FC / 8);
    if (FC == 8) {
      ring[wq & (RING_WORDS - 1)] = f0 | (f1 << 8) | (f2 << 16) | (f3 << 24);
    } else if (FC == 16) {
      ring[wq & (RING_WORDS - 1)] = f0 | (f1 << 16);
      ring[(wq + 1) & (RING_WORDS - 1)] = f2 | (f3 << 16);
    } else {
      ring[wq & (RING_WORDS - 1)] = f0 | (f1 << 24);
      ring[(wq + 1) & (RING_WORDS - 1)] = (f1 >> 8) | (f2 << 16);
      ring[(wq + 2) & (RING_WORDS - 1)] = (f2 >> 16) | (f3 << 8);
    }
  } else {
    wq += pos * 4;
    ring[wq & (RING_WORDS - 1)] = v.x;
    ring[(wq + 1) & (RING_WORDS - 1)] = v.y;
    ring[(wq + 2) & (RING_WORDS - 1)] = v.z;
    ring[(wq + 3) & (RING_WORDS - 1)] = v.w;
  }
  const uint32_t nmatch = __popc(frag);
  sp.pb += (nmatch * MW + ((uint32_t)BPS - nmatch) * (uint32_t)LWB) << 5;
}

// Any other step (the row's last one, or blocks of 8 or 16 lane words).
template <int LWB>
__device__ __forceinline__ void pack_step(const Code &code, const Runs4 &runs,
                                          const SharedRuns &sruns, WarpRing &w,
                                          const uint32_t (&xg)[4], int nw_step, uint32_t frag,
                                          StreamPos &sp, int qh, const PackLane &pl) {
  constexpr int SEG = LWB < 32 ? LWB : 32;
  constexpr int SPG = 32 / SEG;
  const int lane = threadIdx.x & 31;
  const uint32_t fc = (uint32_t)code.fc;
  const uint32_t wq0 = (uint32_t)qh + (sp.pb >> 5);  // stream word of the step's payload
  uint32_t bits = 0;  // payload bits of the step so far (whole words before the last block)
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const int g0 = 32 * g;
    if (g0 >= nw_step) break;
    const int nvg = min(32, nw_step - g0);  // lane words of the row in this group
    const uint32_t x = xg[g];
    const int seg = lane / SEG, kk = lane % SEG;
    // match bits of the group's segments; a block of 64 lane words spans two groups,
    // both carrying its one bit
    const uint32_t segp = LWB > 32 ? ((frag >> (g0 / LWB)) & 1u)
                                   : ((frag >> (g * SPG)) & low_mask((uint32_t)SPG));
    const uint32_t p = (segp >> seg) & 1u;
    uint32_t out = x;
    if (segp != 0u && fc != 0u) {
      const uint32_t c = pack_word<SEG>(extract4(x, runs, sruns), fc, pl);
      if (p) out = c;
    }
    const int nvl = min(SEG, max(0, nvg - seg * SEG));  // lane words of my segment
    const uint32_t words = p ? ((uint32_t)nvl * fc + 31u) >> 5 : (uint32_t)nvl;
    // earlier segments of the group are whole blocks
    const uint32_t mb = __popc(segp & low_mask((uint32_t)seg));
    const uint32_t before = (mb * (uint32_t)SEG * fc + ((uint32_t)seg - mb) * 32u * SEG) >> 5;
    if ((uint32_t)kk < words)
      w.ring()[(wq0 + (bits >> 5) + before + (uint32_t)kk) & (RING_WORDS - 1)] = out;
    for (int s2 = 0; s2 * SEG < nvg; ++s2) {
      const uint32_t n2 = (uint32_t)min(SEG, nvg - s2 * SEG);
      bits += ((segp >> s2) & 1u) ? n2 * fc : 32u * n2;
    }
  }
  sp.pb += bits;
}

// The complete stream vectors [sp.fv, fe) to the slot (sp.fv starts at the vector of
// stream word qh, the first with payload bits; the ones before hold participation
// bits only and are written at the row's end): stream word q is payload word q - qh
// (ring index q) moved up by s0 bits over the top of the word before it (ring words
// below qh read as zero: those bits are participation bits, ORed in at the end). The
// vector below hv that also holds participation bits goes to the warp's head buffer;
// only vectors below nvec are written (a stream that reaches further belongs to a row
// stored raw).
__device__ __forceinline__ void flush(WarpRing &w, uint4 *dst, StreamPos &sp, int fe,
                                      uint32_t s0, int hv, int nvec, int lane) {
  const uint4 *ring4 = reinterpret_cast<const uint4 *>(w.ring());
  for (int v = sp.fv + lane; v < fe; v += 32) {
    const uint4 cur = ring4[v & (RING_VECS - 1)];
    const uint32_t prev = w.ring()[(4 * v - 1) & (RING_WORDS - 1)];
    const uint4 val = make_uint4(__funnelshift_l(prev, cur.x, s0), __funnelshift_l(cur.x, cur.y, s0),
                                 __funnelshift_l(cur.y, cur.z, s0), __funnelshift_l(cur.z, cur.w, s0));
    if (v < hv) *w.head() = val;
    else if (v < nvec) dst[v] = val;
  }
  if (fe > sp.fv) sp.fv = fe;
}

// flush for the vectors a step completes: at most 32, one per lane. sp.fv is the
// vector of stream word qh + pb/32 rounded down (all complete vectors before it are
// out), and a step adds at most 128 payload words, so fe - sp.fv <= 32.
__device__ __forceinline__ void flush_step(WarpRing &w, uint4 *dst, StreamPos &sp, int fe,
                                           uint32_t s0, int hv, int nvec, int lane) {
  const uint4 *ring4 = reinterpret_cast<const uint4 *>(w.ring());
  const int v = sp.fv + lane;
  if (v < fe) {
    const uint4 cur = ring4[v & (RING_VECS - 1)];
    const uint32_t prev = w.ring()[(4 * v - 1) & (RING_WORDS - 1)];
    const uint4 val =
        make_uint4(__funnelshift_l(prev, cur.x, s0), __funnelshift_l(cur.x, cur.y, s0),
                   __funnelshift_l(cur.y, cur.z, s0), __funnelshift_l(cur.z, cur.w, s0));
    if (v < hv) *w.head() = val;
    else if (v < nvec) dst[v] = val;
  }
  if (fe > sp.fv) sp.fv = fe;
}

// FC8 (8, 16 or 24; 0: off): with FAST, full steps are matched and packed from the
// 16-byte view (pack_vec); other steps as below.
template <int LWB, bool FAST, int FC8 = 0>
__device__ void stream_rows(const StreamArgs &a, const Code &code, const SharedRuns &sruns,
                            WarpRing &w) {
  constexpr int BPS = 128 / LWB;  // blocks per step
  constexpr int SEG = LWB < 32 ? LWB : 32;
  const Runs4 runs = load_runs4(sruns);
  const int lane = threadIdx.x & 31;
  const int nvec = a.raw_words >> 2;
  const int nsteps = (nvec + 31) >> 5;
  const int hv = (a.nb + 127) >> 7;  // vectors holding participation bits
  const int qh = a.nb >> 5;          // payload word 0 starts in stream word qh ...
  const uint32_t s0 = (uint32_t)a.nb & 31u;  // ... at this bit
  PackLane pl{0, 0u, 0, 32u, 32u, 0u, 0u};
  if (code.fc > 0) {
    const uint32_t fc = (uint32_t)code.fc;
    const uint32_t kk = (uint32_t)(lane % SEG);
    pl.i0 = (int)(32u * kk / fc);
    pl.a0 = 32u * kk - (uint32_t)pl.i0 * fc;
    pl.nt = (int)(31u / fc) + 2;
    pl.l1 = fc - pl.a0;
    pl.l2 = 2u * fc - pl.a0;
    pl.m1 = pl.l1 < 32u ? 1u << pl.l1 : 0u;
    pl.m2 = pl.l2 < 32u ? 1u << pl.l2 : 0u;
  }
  const int64_t gw = (int64_t)blockIdx.x * SW_WARPS + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * SW_WARPS;
  if (blockIdx.x == 0 && threadIdx.x == 0 && (a.n_rows & 31))
    atomicAnd(&a.bitmask[a.n_rows >> 5], low_mask((uint32_t)(a.n_rows & 31)));
  // every row rewrites each participation-bit word below ceil(nb / 32); the words
  // past it up to the vector boundary are read at the row's end and stay zero
  for (int q = lane; q < a.hdr_words; q += 32) w.hdr()[q] = 0u;
  for (int64_t r = gw; r < a.n_rows; r += nwarps) {
    const uint4 *src = reinterpret_cast<const uint4 *>(a.rows + r * a.raw_bytes);
    uint4 *dst = reinterpret_cast<uint4 *>(a.slots + r * a.slot_bytes);
    // the first flushed vector (that of stream word qh) reads the ring words from the
    // one before it up to qh - 1: they stand for participation bits and read as zero;
    // every later word the flush reads is written by this row first
    if (lane < 4) {
      const int q = 4 * (qh >> 2) - 1 + lane;
      if (q < qh) w.ring()[q & (RING_WORDS - 1)] = 0u;
    }
    __syncwarp();
    StreamPos sp{0u, qh >> 2};
    bool streaming = false;  // false: no block has matched yet, vectors copied raw
    int k_seen = 0;          // steps whose match bits are in the header
    uint32_t hcur = 0;       // participation-bit word being filled
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
      for (int i = 0; i < PF - 1; ++i) {
        if (32 * i + lane < nvec) cp_async16(&w.stage()[i][lane], src + 32 * i + lane);
        cp_async_commit();
      }
      bool restart = false;
#pragma unroll 1
      for (int k = 0; k < nsteps; ++k) {
        {
          const int kn = k + PF - 1, vn = 32 * kn + lane;  // into the slot step k - 1 used
          if (vn < nvec) cp_async16(&w.stage()[kn % PF][lane], src + vn);
          cp_async_commit();
        }
        cp_async_wait<PF - 1>();  // this lane's copy of step k has landed
        __syncwarp();             // ... and every other lane's
        const int nw_step = min(128, a.raw_words - 128 * k);
        uint32_t *S = reinterpret_cast<uint32_t *>(&w.stage()[k % PF][0]);
        uint32_t xg[4];
        uint4 v4;
        const bool vec = FC8 != 0 && nw_step == 128;  // a full step (no partial block)
        const int b0 = k * BPS;
        uint32_t frag;
        if (vec) {
          v4 = w.stage()[k % PF][lane];
          frag = vec_frag<LWB>(v4, code);
        } else {
          if (nw_step == 128) {
#pragma unroll
            for (int g = 0; g < 4; ++g) xg[g] = S[32 * g + lane];
          } else {
#pragma unroll
            for (int g = 0; g < 4; ++g) xg[g] = 32 * g + lane < nw_step ? S[32 * g + lane] : 0u;
          }
          frag = group_frag<LWB>(xg, nw_step, min(BPS, a.nb - b0), code);
        }
        if (k >= k_seen) {
          hcur |= frag << (b0 & 31);
          if (((b0 + BPS) & 31) == 0 || k == nsteps - 1) {
            if (lane == 0) w.hdr()[b0 >> 5] = hcur;
            hcur = 0;
          }
          k_seen = k + 1;
        }
        if (!streaming) {
          if (frag == 0) {  // still no match in the row: copy the vector raw
            const int v = 32 * k + lane;
            if (v < nvec) dst[v] = w.stage()[k % PF][lane];
            __syncwarp();  // the others read this slot; the next step's copies reuse it
            continue;
          }
          streaming = true;  // first matching block: start over in stream mode
          restart = true;
          cp_async_wait<0>();  // no copy into the staging slots is left in flight
          __syncwarp();
          break;
        }
        if constexpr (FC8 != 0) {
          if (vec) {
            pack_vec<LWB, (FC8 ? FC8 : 8)>(runs, w, v4, frag, sp, qh);
          } else {
            pack_step<LWB>(code, runs, sruns, w, xg, nw_step, frag, sp, qh, pl);
          }
        } else if (LWB >= 32 && nw_step == 128) {
          pack_full<LWB, FAST>(code, runs, sruns, w, xg, frag, sp, qh, pl);
        } else {
          pack_step<LWB>(code, runs, sruns, w, xg, nw_step, frag, sp, qh, pl);
        }
        __syncwarp();
        flush_step(w, dst, sp, (int)(((uint32_t)qh + (sp.pb >> 5)) >> 2), s0, hv, nvec, lane);
        __syncwarp();
      }
      if (!restart) break;
    }
    cp_async_wait<0>();
    // the row's size and the raw-or-compressed decision (a row that never matched is
    // nb bits longer than raw)
    const uint32_t total = (uint32_t)a.nb + (streaming ? sp.pb : 32u * (uint32_t)a.raw_words);
    const uint32_t sw = (total + 31) >> 5;
    const bool comp = (int64_t)sw * 4 < a.raw_bytes;  // implies streaming
    if (comp) {
      // payload words past the last one read as zeros, then the rest of the stream
      if (lane < 8)
        w.ring()[((uint32_t)qh + ((sp.pb + 31) >> 5) + (uint32_t)lane) & (RING_WORDS - 1)] = 0u;
      __syncwarp();
      flush(w, dst, sp, (int)((sw + 3) >> 2), s0, hv, nvec, lane);
      __syncwarp();
      // the vectors holding participation bits: those before the first payload word
      // are the bits alone, the one shared with the payload gets them ORed in
      const uint4 *hdr4 = reinterpret_cast<const uint4 *>(w.hdr());
      for (int v = lane; v < hv; v += 32) {
        uint4 h = hdr4[v];
        if (v >= (qh >> 2)) {
          const uint4 p = *w.head();
          h = make_uint4(h.x | p.x, h.y | p.y, h.z | p.z, h.w | p.w);
        }
        dst[v] = h;
      }
    } else if (streaming) {  // matched somewhere but saves nothing: store the row raw
      for (int v = lane; v < nvec; v += 32) dst[v] = load_vec(src + v);
    }
    if (lane == 0) {
      if (a.row_bits) a.row_bits[r] = total;
      const uint32_t bit = 1u << (r & 31);
      if (comp) atomicOr(&a.bitmask[r >> 5], bit);
      else atomicAnd(&a.bitmask[r >> 5], ~bit);
    }
    __syncwarp();
  }
}

template <int LWB>
__global__ void __launch_bounds__(SW_THREADS, SW_CTAS_PER_SM) compress_stream_kernel(StreamArgs a) {
  extern __shared__ __align__(16) uint8_t smem_stream[];
  __shared__ SharedRuns sruns;
  const ibp_meta m = load_meta(a.meta);
  if (m.dtype != a.dtype || m.block_elems != a.block_elems) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(a.status, IBP_ERR_META);
    return;
  }
  const Code code = make_code(m);
  if (threadIdx.x == 0) make_runs(~code.mask32, sruns);
  __syncthreads();
  WarpRing w;
  w.base = smem_stream + (threadIdx.x >> 5) * warp_ring_bytes(a.hdr_words);
  // the common masks (at most four runs of kept bits, bit 0 kept) get their own copies
  // of the row loop: fields of 8, 16 or 24 bits (whole words per four fields), other
  // fields of at least 16 bits; only one copy runs in a launch
  const bool fast_runs = sruns.n <= 4 && sruns.n > 0 && sruns.sh[0] == 0u;
  if (fast_runs && code.fc == 24)
    stream_rows<LWB, true, 24>(a, code, sruns, w);
  else if (fast_runs && code.fc == 16)
    stream_rows<LWB, true, 16>(a, code, sruns, w);
  else if (fast_runs && code.fc == 8)
    stream_rows<LWB, true, 8>(a, code, sruns, w);
  else if (fast_runs && code.fc >= 16)
    stream_rows<LWB, true>(a, code, sruns, w);
  else
    stream_rows<LWB, false>(a, code, sruns, w);
}

template <int LWB>
int launch_stream(const StreamArgs &a, const DeviceInfo &dev, cudaStream_t s) {
  // the largest dynamic size, leaving room for the kernel's static shared memory
  const int dyn_max = dev.max_smem_optin - (int)sizeof(SharedRuns) - 1024;
  const size_t smem = warp_ring_bytes(a.hdr_words) * SW_WARPS;
  if (smem > (size_t)dyn_max) return IBP_ERR_UNSUPPORTED;
  static std::atomic<int> configured[64];  // the attribute is set once per device
  if (dev.device >= 64 || !configured[dev.device].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(compress_stream_kernel<LWB>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max) != cudaSuccess)
      return IBP_ERR_CUDA;
    if (dev.device < 64) configured[dev.device].store(1, std::memory_order_release);
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, compress_stream_kernel<LWB>,
                                                    SW_THREADS, smem) != cudaSuccess ||
      per_sm < 1)
    return IBP_ERR_CUDA;
  const int64_t want = (a.n_rows + SW_WARPS - 1) / SW_WARPS;
  const int grid = (int)std::min<int64_t>(want, (int64_t)dev.sm_count * per_sm);
  compress_stream_kernel<LWB><<<grid, SW_THREADS, smem, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

}  // namespace

int launch_compress_stream(const void *rows, int64_t n_rows, const RowGeom &g, uint32_t dtype,
                           const ibp_meta *d_meta, void *slots, int64_t slot_bytes,
                           uint32_t *d_bitmask, uint32_t *d_row_bits, int32_t *d_status,
                           const DeviceInfo &dev, cudaStream_t s) {
  if (g.raw_words % 4 != 0) return IBP_ERR_UNSUPPORTED;
  StreamArgs a;
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
  a.raw_bytes = g.raw_bytes;
  a.hdr_words = ((g.nb + 31) / 32 + 3) & ~3;
  switch (g.lwb) {
    case 8: return launch_stream<8>(a, dev, s);
    case 16: return launch_stream<16>(a, dev, s);
    case 32: return launch_stream<32>(a, dev, s);
    default: return launch_stream<64>(a, dev, s);
  }
}

}  // namespace ibp
