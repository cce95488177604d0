// Decompress-gather kernel of Invariant Bit Packing for sm_103a.
//
// "Reducing the GPU Memory Bottleneck with Lossless Compression for ML --
// Extended", technical summary, "Core algorithm" (decompression) and "System
// integration" (fixed-size buffers of which only the compressed part is read,
// GPU-resident bitmask of compressed rows).
//
// Work unit: one segment (at most 32 consecutive blocks) of one requested row.
// A team of TL lanes (TL = 4..32, chosen so each lane rebuilds a few 16-byte
// vectors) owns one unit at a time; a warp runs 32/TL teams side by side, so no
// per-unit broadcast is needed. Every lane of a team:
//   1. plans the unit: index -> bitmask bit -> participation bits of the row
//      header (the same words for the whole team, one request). Population
//      counts of the header words give the number of compressed blocks before
//      the segment and with it the segment's first bit: the prefix scan of
//      block sizes reduces to a popcount because a block is either B*m or B*w
//      bits long;
//   2. stages its share of the 16-byte-aligned span of the slot that holds the
//      segment into shared memory with cp.async (L1-coalesced, so each 128-byte
//      line is requested once; works for HBM and for registered host memory
//      read zero-copy over the host link);
//   3. rebuilds 4 lane words (16 output bytes) per step without branches: block
//      of the vector, its participation bit, popcount of the earlier bits ->
//      bit position; funnel-shift each field out of shared memory, deposit it
//      over the non-invariant positions of bitval; 128-bit store.
// Packed stores (rows end to end, entry r at offsets[r], 16-byte aligned): the
// row's entry length comes with its offset, so a one-segment row is staged whole,
// exactly its stored bytes, without reading its header first.
// The loop is software-pipelined two deep: the next unit's plan and staging are
// issued before the current unit is decoded, and the index two units ahead is
// prefetched, so header and body round trips overlap with decode.
// De-duplicated gathers of rows that are one unit each use a claiming instantiation
// (CLAIM): before a unit is planned its leader claims the row in a hash table, and
// only the first claimant stages and decodes it (ibp_dedup.cu copies the rest).
#include <algorithm>
#include <atomic>

#include "ibp_device.cuh"
#include "ibp_internal.h"

namespace ibp {
namespace {

constexpr int GATHER_WARPS = 4;         // warps per CTA (measured: 2-3 % faster than 8 on HBM)
constexpr int GATHER_NBUF = 2;          // staging buffers per team (units in flight + 1)
constexpr int SEG_TARGET_BYTES = 4096;  // raw bytes per segment (at most 32 blocks)

struct GatherArgs {
  const uint8_t *slots;      // slotted store, or the packed store's bytes
  int64_t slot_bytes;        // slotted store only
  const uint64_t *offsets;   // packed store: entry offsets [n_rows + 1]; null if slotted
  const uint32_t *row_bits;  // slotted store with known row sizes (sized gather), or null
  uint64_t packed_bytes;     // packed or sized: bytes of the buffer at slots
  int64_t n_rows;
  const uint32_t *bitmask;
  const ibp_meta *meta;
  const int64_t *idx;  // null: rows row0, row0 + 1, ... in order
  int64_t row0;
  int64_t n_idx;
  uint32_t *out;
  int32_t *status;
  uint32_t dtype, block_elems;
  int lwb, lwb_shift, nb, raw_words;
  int lwt;  // lane words of the last block (lwb, or fewer for a shorter tail)
  int seg_blocks, nseg;
  int unit_bytes;  // shared staging bytes per unit (one buffer)
  int64_t n_units;
  int64_t raw_bytes;
  int cta0, ncta;  // the CTAs [cta0, cta0 + ncta) of the grid work on this gather
  // Sized gather: the staged prefix of a slot ends on a multiple of this many bytes
  // of the address space (within the slot). Packed store: the staged bytes start and
  // end on such multiples (within the store and the staging buffer) around the entry.
  // 128 for host memory, where a partly read 128-byte line costs the link about as
  // much as a whole one; 16 for HBM.
  uint32_t span_align;
  // a negative index is a unit with nothing to do, not an error (internal lists whose
  // tail is unused, e.g. the distinct rows of a de-duplicated gather)
  uint32_t skip_negative;
  // index entries carry the output row of their unit in bits 40..63 and the row in
  // bits 0..39 (the compact list of a de-duplicated gather: each distinct row is
  // decoded straight into the first output row that asks for it)
  uint32_t pos_in_index;
  // number of index entries to gather, read on the device when the kernel starts
  // (null: all n_idx); entries past it are not even looked at
  const unsigned long long *idx_count;
  // limit of each bounded wait of the warp-specialised kernel, in ns of global time
  uint64_t wait_ns;
  // de-duplicated gather of rows that are one unit each (null table: off): before a
  // unit is planned its position claims the row in this hash table; only the first
  // claimant decodes it, claim_owner[position] receives the claimant
  unsigned long long *claim_table;
  uint32_t claim_mask;
  int32_t *claim_owner;
  // testing hook: the warp-specialised kernel's planners never hand a plan over
  uint32_t withhold_plans;
};

// The plan of one unit (identical in every lane of its team).
struct Unit {
  const uint8_t *src;  // first staged byte
  int64_t out_word;    // first output lane word of the segment
  uint32_t nchunk;     // 16-byte chunks to stage (0: nothing to do)
  uint32_t nvec;       // 16-byte output vectors (0: nothing to do)
  uint32_t lsb;        // bit offset of the segment's first block in the staged bytes
  uint32_t segp;       // participation bits of the segment's blocks (0 for raw rows);
                       // the row index when lsb == PARSE_HEADER
  uint32_t bmw;        // bitmask word of the row (only when lsb == PARSE_HEADER)
  uint32_t echunk;     // packed entry or sized span: its 16-byte chunks (checks)
  uint32_t lead;       // staged bytes in front of the entry (whole-line staging)
};

// Unit.lsb value telling the decoder to take the participation bits from the
// staged bytes (the whole slot prefix was staged).
constexpr uint32_t PARSE_HEADER = 0xFFFFFFFFu;

// Stage whole slots (one round trip less per compressed row) when compression can
// save at most a fifth of a row: even a row whose blocks all match then stores at
// least 80% of its raw bytes, so reading the raw-size prefix costs little extra.
// Rows of one segment only (the participation bits then fit one word).
__device__ __forceinline__ bool whole_slot(const GatherArgs &a, uint32_t shrink) {
  const uint32_t fc = 32u - shrink;
  const uint32_t min_bits = (uint32_t)a.nb + (uint32_t)a.lwb * (uint32_t)a.nb * fc;
  return (int64_t)((min_bits + 31) >> 5) * 4 * 5 >= a.raw_bytes * 4;
}

// Units to gather: all of them, or those of the first *idx_count index entries.
__device__ __forceinline__ int64_t units_of(const GatherArgs &a) {
  if (!a.idx_count) return a.n_units;
  const int64_t c = (int64_t)*a.idx_count * a.nseg;
  return c < a.n_units ? c : a.n_units;
}

__device__ __forceinline__ int64_t load_index(const GatherArgs &a, int64_t u, int64_t n_units) {
  if (u >= n_units) return -1;
  const int64_t i = a.nseg == 1 ? u : u / a.nseg;
  return a.idx ? __ldg(a.idx + i) : a.row0 + i;
}

// The claim of unit u's row (a row of one unit, so u is the output position) for a
// de-duplicated gather, by one lane per unit. The table maps row + 1 to the first
// position that claimed it, both in one 64-bit word (row in the top 40 bits), set by
// one compare-and-swap; a row claimed earlier is usually seen by a plain L2 load,
// without an atomic. Returns r for the claimant (it decodes the row) and -1 for every
// other position (nothing to stage; the copy comes later) and for a bad index
// (reported here). claim_owner[u] receives the claimant, or -1 for a bad index.
constexpr int CLAIM_POS_BITS = 24;

__device__ int64_t claim_row(const GatherArgs &a, int64_t u, int64_t n_units, int64_t r) {
  if (u >= n_units) return r;
  if (r < 0 || r >= a.n_rows) {
    a.claim_owner[u] = -1;
    report(a.status, IBP_ERR_INDEX);
    return -1;
  }
  const unsigned long long key = (unsigned long long)r + 1ull;
  const unsigned long long mine = (key << CLAIM_POS_BITS) | (unsigned long long)u;
  uint32_t h = (uint32_t)((key * 0x9E3779B97F4A7C15ull) >> 32) & a.claim_mask;  // Fibonacci
  int32_t own = -1;
  // at least two slots per position: a free slot or the row's entry is found within
  // mask + 1 probes
  for (uint32_t probe = 0; probe <= a.claim_mask; ++probe) {
    unsigned long long old = __ldcg(a.claim_table + h);
    if (old == 0ull) old = atomicCAS(a.claim_table + h, 0ull, mine);
    if (old == 0ull) {
      own = (int32_t)u;
      break;
    }
    if ((old >> CLAIM_POS_BITS) == key) {
      own = (int32_t)(old & ((1ull << CLAIM_POS_BITS) - 1));
      break;
    }
    h = (h + 1) & a.claim_mask;
  }
  a.claim_owner[u] = own;
  return own == (int32_t)u ? r : -1;
}

// The bytes of row r to stage, [o0, o1) of the buffer at slots: a packed store's
// entry, or (sized gather) the used prefix of the row's slot from its bitmask bit
// and bit count, extended to an address that is a multiple of span_align (16 or
// 128) and cut at the slot's end. Both 0 for a bad index.
struct EntrySpan {
  uint64_t o0, o1;
};

__device__ __forceinline__ EntrySpan load_span(const GatherArgs &a, int64_t r) {
  EntrySpan e{0, 0};
  if (r < 0 || r >= a.n_rows) return e;
  if (a.offsets) {
    e.o0 = __ldg(a.offsets + r);
    e.o1 = __ldg(a.offsets + r + 1);
  } else if (a.row_bits) {
    const uint32_t bits = __ldg(a.row_bits + r);
    const bool comp = (__ldg(a.bitmask + (r >> 5)) >> (r & 31)) & 1u;
    const uint64_t used = comp ? 4ull * (((uint64_t)bits + 31) >> 5) : (uint64_t)a.raw_bytes;
    const uint64_t slot = (uint64_t)a.slot_bytes;
    e.o0 = (uint64_t)r * slot;
    const uint64_t base = (uint64_t)(uintptr_t)a.slots;
    const uint64_t al = a.span_align;
    const uint64_t len = ((base + e.o0 + used + al - 1) & ~(al - 1)) - (base + e.o0);
    e.o1 = e.o0 + (len < slot ? len : slot);
  }
  return e;
}

// PACKED: the bytes to stage come with the row (a packed store's entry, or a sized
// gather's used slot prefix); span: those bytes, loaded ahead by the caller. The
// plain slotted instantiation carries none of it.
template <bool PACKED>
__device__ __forceinline__ Unit plan_unit(const GatherArgs &a, uint32_t shrink, int64_t u,
                                          int64_t n_units, int64_t r, bool leader,
                                          EntrySpan span) {
  Unit un;
  un.src = a.slots;
  un.out_word = 0;
  un.nchunk = 0;
  un.nvec = 0;
  un.lsb = 0;
  un.segp = 0;
  un.bmw = 0;
  un.echunk = 0;
  un.lead = 0;
  if (u >= n_units) return un;
  int64_t i = u;
  int s = 0;
  if (a.nseg != 1) {
    i = u / a.nseg;
    s = (int)(u - i * a.nseg);
  }
  const int b0 = s * a.seg_blocks;
  const int nblk = min(a.seg_blocks, a.nb - b0);
  if (a.pos_in_index && r >= 0) {
    i = r >> 40;
    r &= (int64_t(1) << 40) - 1;
  }
  un.out_word = i * (int64_t)a.raw_words + (int64_t)b0 * a.lwb;
  if (r < 0 || r >= a.n_rows) {
    if (leader && !(a.skip_negative && r < 0)) report(a.status, IBP_ERR_INDEX);
    return un;
  }
  const bool last_seg = b0 + nblk == a.nb;  // holds the row's last block
  const uint32_t seg_words = (uint32_t)(nblk * a.lwb - (last_seg ? a.lwb - a.lwt : 0));
  const uint32_t nvec = seg_words / 4;
  const uint8_t *slot;
  int64_t avail;  // readable bytes of the row's slot or entry
  if (PACKED) {
    const uint64_t o0 = span.o0, o1 = span.o1;
    if (o1 < o0 || (o0 & 15) || (o1 & 15) || o1 > a.packed_bytes) {
      if (leader) report(a.status, IBP_ERR_CORRUPT);
      return un;
    }
    slot = a.slots + o0;
    avail = (int64_t)(o1 - o0);
  } else {
    slot = a.slots + r * a.slot_bytes;
    avail = a.slot_bytes;
  }
  if (a.nseg == 1 && a.n_rows <= 0xFFFFFFFFll && (PACKED || whole_slot(a, shrink))) {
    // stage the slot's whole raw-size prefix (a packed entry: all of it) at once:
    // the bitmask bit and, for a compressed row, the participation bits are read
    // later, off the critical path
    un.src = slot;
    un.nchunk = PACKED ? (uint32_t)min((int64_t)nvec, avail >> 4) : nvec;
    un.echunk = un.nchunk;
    un.nvec = nvec;
    un.lsb = PARSE_HEADER;
    un.segp = (uint32_t)r;
    if (PACKED && a.offsets && a.span_align > 16) {
      // whole lines around the entry: from the line it starts in to the end of the
      // line it ends in, inside the store and leaving the staging buffer room for
      // the decoder's look-ahead word
      const uint64_t al = a.span_align;
      const uint64_t base = (uint64_t)(uintptr_t)a.slots;
      const uint64_t e0 = base + span.o0;
      uint64_t s0 = e0 & ~(al - 1);
      if (s0 < base) s0 = base;
      uint64_t s1 = (base + span.o1 + al - 1) & ~(al - 1);
      if (s1 > base + a.packed_bytes) s1 = base + a.packed_bytes;
      const uint64_t cap = (uint64_t)a.unit_bytes - 16;
      if (e0 - s0 + 16ull * un.echunk <= cap) {
        if (s1 - s0 > cap) s1 = s0 + cap;
        un.src = a.slots + (s0 - base);
        un.lead = (uint32_t)(e0 - s0);
        un.nchunk = (uint32_t)((s1 - s0) >> 4);
      }
    }
    return un;
  }
  if (!((__ldg(a.bitmask + (r >> 5)) >> (r & 31)) & 1u)) {  // stored raw
    if (PACKED && avail < a.raw_bytes) {
      if (leader) report(a.status, IBP_ERR_CORRUPT);
      return un;
    }
    un.src = slot + (size_t)b0 * a.lwb * 4;
    un.nchunk = nvec;
    un.nvec = nvec;
    return un;
  }
  // participation bits: nb bits at the start of the slot
  const uint32_t *hw = reinterpret_cast<const uint32_t *>(slot);
  const int nhw = (a.nb + 31) >> 5;
  if (PACKED && avail < 4 * nhw) {
    if (leader) report(a.status, IBP_ERR_CORRUPT);
    return un;
  }
  uint32_t cnt_all = 0, cnt0 = 0, lo = 0, hi = 0, p_last = 0;
  const int q0 = b0 >> 5;
  for (int q = 0; q < nhw; ++q) {
    uint32_t word = hw[q];
    if (q == q0) lo = word;
    if (q == q0 + 1) hi = word;
    if (q == nhw - 1) {
      word &= low_mask((uint32_t)(a.nb - 32 * q));
      p_last = (word >> ((a.nb - 1) & 31)) & 1u;
    }
    const uint32_t c = __popc(word);
    cnt_all += c;
    if (32 * q + 32 <= b0) cnt0 += c;
    else if (32 * q < b0) cnt0 += __popc(word & low_mask((uint32_t)(b0 - 32 * q)));
  }
  if (q0 + 1 >= nhw) hi = 0;
  const uint32_t segp = window(lo, hi, (uint32_t)(b0 & 31)) & low_mask((uint32_t)nblk);
  // bits = nb + sum over blocks of lane words * (p ? fc : 32); the last block has
  // lwt lane words, every other one lwb
  const uint32_t short_last = (uint32_t)(a.lwb - a.lwt) * p_last;
  const uint32_t total = (uint32_t)a.nb + 32u * (uint32_t)a.raw_words -
                         shrink * ((uint32_t)a.lwb * cnt_all - short_last);
  const int64_t used = (int64_t)((total + 31) >> 5) * 4;
  if (used >= a.raw_bytes || (PACKED && used > avail)) {
    if (leader) report(a.status, IBP_ERR_CORRUPT);
    return un;
  }
  const uint32_t st = (uint32_t)a.nb + (uint32_t)a.lwb * (32u * (uint32_t)b0 - shrink * cnt0);
  const uint32_t en = st + 32u * seg_words -
                      shrink * ((uint32_t)a.lwb * __popc(segp) - (last_seg ? short_last : 0u));
  const uint32_t w0 = (st >> 5) & ~3u;
  const uint32_t w1 = ((en + 127) >> 7) << 2;
  un.src = slot + (size_t)w0 * 4;
  un.nchunk = (w1 - w0) >> 2;
  un.nvec = nvec;
  un.lsb = st - 32 * w0;
  un.segp = segp;
  return un;
}

// Issue the bitmask load of a whole-slot unit; its value is used one pipeline step
// later, when the unit is decoded.
__device__ __forceinline__ void fetch_bitmask(const GatherArgs &a, Unit &un) {
  if (un.lsb == PARSE_HEADER) un.bmw = __ldg(a.bitmask + (un.segp >> 5));
}

template <int TL>
__device__ __forceinline__ void stage_unit(const Unit &un, uint8_t *buf, int tl) {
  for (uint32_t c = tl; c < un.nchunk; c += TL) cp_async16(buf + 16 * c, un.src + 16 * c);
}

template <int NR, int TL, bool PACKED>
__device__ __forceinline__ void decode_unit(const GatherArgs &a, const Code &code,
                                            const RegRuns<NR> &runs, const SharedRuns &sruns,
                                            const Unit &un, const uint8_t *buf, int tl) {
  // the staged bytes start un.lead bytes before the entry (whole-line staging)
  const uint32_t fc = (uint32_t)code.fc;
  const uint32_t shrink = 32u - fc;
  buf += un.lead;
  const uint32_t *S = reinterpret_cast<const uint32_t *>(buf);
  uint4 *dst = reinterpret_cast<uint4 *>(a.out + un.out_word);
  uint32_t segp = un.segp, lsb = un.lsb, nvec = un.nvec;
  if (lsb == PARSE_HEADER) {  // whole slot (or packed entry) staged, un.nchunk pieces
    if (!((un.bmw >> (segp & 31)) & 1u)) {  // stored raw: the slot prefix is the row
      segp = 0;
      lsb = 0;
      if (PACKED && un.echunk < nvec) {  // a packed entry shorter than the raw row
        if (tl == 0) report(a.status, IBP_ERR_CORRUPT);
        nvec = 0;
      }
    } else {  // participation bits are S[0] (one segment, nb <= 32)
      segp = (!PACKED || un.echunk) ? (S[0] & low_mask((uint32_t)a.nb)) : 0u;
      lsb = (uint32_t)a.nb;
      const uint32_t p_last = (segp >> (a.nb - 1)) & 1u;
      const uint32_t total =
          (uint32_t)a.nb + 32u * (uint32_t)a.raw_words -
          shrink * ((uint32_t)a.lwb * __popc(segp) - (uint32_t)(a.lwb - a.lwt) * p_last);
      const int64_t used = (int64_t)((total + 31) >> 5) * 4;
      if (used >= a.raw_bytes || (PACKED && used > 16 * (int64_t)un.echunk)) {
        if (tl == 0) report(a.status, IBP_ERR_CORRUPT);
        nvec = 0;
      }
    }
  }
  if (segp == 0 && lsb == 0) {  // row stored raw: the staged bytes are the row
    const uint4 *S4 = reinterpret_cast<const uint4 *>(buf);
    for (uint32_t v = tl; v < nvec; v += TL) dst[v] = S4[v];
    return;
  }
  for (uint32_t v = tl; v < nvec; v += TL) {
    const uint32_t lw = 4 * v;
    const uint32_t lb = lw >> a.lwb_shift;
    const uint32_t j = lw - (lb << a.lwb_shift);  // lane word within its block
    const uint32_t cnt = __popc(segp & low_mask(lb));
    const uint32_t blk = lsb + (uint32_t)a.lwb * (32u * lb - shrink * cnt);  // block start bit
    uint4 y;
    if (!((segp >> lb) & 1u)) {
      // block kept raw: four whole words behind one constant bit shift
      const uint32_t pos = blk + 32u * j;
      const uint32_t *w = S + (pos >> 5);
      const uint32_t sh = pos & 31u;
      y.x = window(w[0], w[1], sh);
      y.y = window(w[1], w[2], sh);
      y.z = window(w[2], w[3], sh);
      y.w = window(w[3], w[4], sh);
    } else {
      // matching block: fields of fc bits, invariant bits put back from bitval
      uint32_t pos = blk + j * fc;
      uint32_t f[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t *w = S + (pos >> 5);
        f[t] = deposit_into<NR>(window(w[0], w[1], pos & 31u), code.bitval32, runs, sruns);
        pos += fc;
      }
      y = make_uint4(f[0], f[1], f[2], f[3]);
    }
    dst[v] = y;
  }
}

// Decode one unit with the deposit specialised for the run count of the kept bits
// (warp-uniform branch, once per unit). Only this step is compiled once per run
// count; the pipeline around it exists once, which keeps the kernel's code small
// enough for the instruction cache (one pipeline copy per run count was measured
// 16% slower on 512-byte rows in HBM).
template <int TL, bool PACKED>
__device__ __forceinline__ void decode_dispatch(const GatherArgs &a, const Code &code,
                                                const SharedRuns &sruns, uint32_t nr,
                                                const Unit &un, const uint8_t *buf, int tl) {
  switch (nr) {
    case 0: decode_unit<0, TL, PACKED>(a, code, load_runs<0>(sruns), sruns, un, buf, tl); break;
    case 1: decode_unit<1, TL, PACKED>(a, code, load_runs<1>(sruns), sruns, un, buf, tl); break;
    case 2: decode_unit<2, TL, PACKED>(a, code, load_runs<2>(sruns), sruns, un, buf, tl); break;
    case 3: decode_unit<3, TL, PACKED>(a, code, load_runs<3>(sruns), sruns, un, buf, tl); break;
    case 4: decode_unit<4, TL, PACKED>(a, code, load_runs<4>(sruns), sruns, un, buf, tl); break;
    default: decode_unit<-1, TL, PACKED>(a, code, load_runs<-1>(sruns), sruns, un, buf, tl); break;
  }
}

// Decode-time fields of a staged unit, kept in shared memory next to its buffer.
struct __align__(16) StagedMeta {
  int64_t out_word;
  uint32_t lsb, segp, nvec, bmw, nchunk, lead;  // nchunk, lead: Unit.echunk, Unit.lead
};

// CLAIM (slotted stores only): the de-duplicated gather's claiming mode.
template <int TL, bool PACKED, bool CLAIM = false>
__device__ void gather_body(const GatherArgs &a, const Code &code, const SharedRuns &sruns,
                            uint8_t *warp_smem, StagedMeta *warp_meta) {
  static_assert(!(PACKED && CLAIM), "claims are made on slotted stores only");
  constexpr int TPW = 32 / TL;  // teams per warp
  const uint32_t nr = sruns.n;
  const int lane = threadIdx.x & 31;
  const int team = lane / TL;
  const int tl = lane % TL;
  const bool leader = tl == 0;
  const uint32_t shrink = 32u - (uint32_t)code.fc;
  const int64_t warp_gid = (int64_t)(blockIdx.x - a.cta0) * GATHER_WARPS + (threadIdx.x >> 5);
  const int64_t stride = (int64_t)a.ncta * GATHER_WARPS * TPW;  // between a team's units
  uint8_t *const bufs = warp_smem + team * a.unit_bytes;  // buffer k at bufs + k * buf_step
  const int buf_step = TPW * a.unit_bytes;
  StagedMeta *const metas = warp_meta + team;  // meta k at metas[k * TPW]

  const int64_t n_units = units_of(a);
  int64_t base = warp_gid * TPW;  // first unit of this warp in the current iteration
  if (base >= n_units) return;
  int64_t u_plan = base + team;  // next unit this team plans
  int64_t r_plan = load_index(a, u_plan, n_units);
  // packed stores: the unit after next's index and the next unit's entry span are
  // loaded one step ahead, so neither dependent load waits in front of staging
  int64_t r_next = PACKED ? load_index(a, u_plan + stride, n_units) : -1;
  EntrySpan span_plan = PACKED ? load_span(a, r_plan) : EntrySpan{0, 0};
  int k_plan = 0;                // buffer it goes to
  uint32_t pend_bmw = 0;         // bitmask word loaded for the last planned unit,
  int pend_k = -1;               // stored into its meta one step later

  // plan one unit, stage its bytes, record what decoding it will need
  auto plan_and_stage = [&]() {
    int64_t r_after;
    EntrySpan span_after{0, 0};
    if (PACKED) {
      r_after = load_index(a, u_plan + 2 * stride, n_units);  // prefetch, two units ahead
      span_after = load_span(a, r_next);            // the next unit's entry
    } else {
      r_after = load_index(a, u_plan + stride, n_units);  // prefetch
    }
    if (CLAIM) {  // the team's leader claims, the team follows
      const int64_t rc = leader ? claim_row(a, u_plan, n_units, r_plan) : 0;
      r_plan = __shfl_sync(FULL, rc, lane & ~(TL - 1));
    }
    const Unit un = plan_unit<PACKED>(a, shrink, u_plan, n_units, r_plan, leader, span_plan);
    if (leader && pend_k >= 0) metas[pend_k * TPW].bmw = pend_bmw;
    pend_bmw = un.lsb == PARSE_HEADER ? __ldg(a.bitmask + (un.segp >> 5)) : 0u;
    pend_k = k_plan;
    if (leader) {
      StagedMeta m;
      m.out_word = un.out_word;
      m.lsb = un.lsb;
      m.segp = un.segp;
      m.nvec = un.nvec;
      m.bmw = 0;
      m.nchunk = PACKED ? un.echunk : 0u;
      m.lead = PACKED ? un.lead : 0u;
      metas[k_plan * TPW] = m;
    }
    stage_unit<TL>(un, bufs + k_plan * buf_step, tl);
    cp_async_commit();
    k_plan = k_plan + 1 == GATHER_NBUF ? 0 : k_plan + 1;
    u_plan += stride;
    if (PACKED) {
      r_plan = r_next;
      r_next = r_after;
      span_plan = span_after;
    } else {
      r_plan = r_after;
    }
  };

#pragma unroll 1
  for (int j = 0; j < GATHER_NBUF - 1; ++j) plan_and_stage();
  int k_dec = 0;
  for (;;) {
    plan_and_stage();
    cp_async_wait<GATHER_NBUF - 1>();
    __syncwarp();
    const StagedMeta m = metas[k_dec * TPW];
    Unit un;
    un.src = nullptr;
    un.nchunk = 0u;
    un.echunk = PACKED ? m.nchunk : 0u;
    un.lead = PACKED ? m.lead : 0u;
    un.out_word = m.out_word;
    un.lsb = m.lsb;
    un.segp = m.segp;
    un.nvec = m.nvec;
    un.bmw = m.bmw;
    decode_dispatch<TL, PACKED>(a, code, sruns, nr, un, bufs + k_dec * buf_step, tl);
    __syncwarp();
    base += stride;
    if (base >= n_units) break;
    k_dec = k_dec + 1 == GATHER_NBUF ? 0 : k_dec + 1;
  }
  cp_async_wait<0>();
}


// shared bytes of one warp of the team kernel
__host__ __device__ inline size_t team_warp_bytes(int tl, int unit_bytes) {
  return (size_t)GATHER_NBUF * (32 / tl) * (unit_bytes + sizeof(StagedMeta));
}

// MINB: resident 8-warp equivalents per SM the register budget is sized for (4 for
// slots in device memory, 3 for host memory; measured best for each): with CTAs of
// GATHER_WARPS warps, MINB * 8 / GATHER_WARPS CTAs.
template <int TL, bool PACKED, bool CLAIM = false>
__device__ __forceinline__ void team_gather(const GatherArgs &a, uint8_t *smem,
                                            SharedRuns &sruns) {
  const ibp_meta m = load_meta(a.meta);
  if (m.dtype != a.dtype || m.block_elems != a.block_elems) {
    if ((int)blockIdx.x == a.cta0 && threadIdx.x == 0) report(a.status, IBP_ERR_META);
    return;
  }
  const Code code = make_code(m);
  if (threadIdx.x == 0) make_runs(~code.mask32, sruns);
  __syncthreads();
  uint8_t *warp_smem = smem + (threadIdx.x >> 5) * team_warp_bytes(TL, a.unit_bytes);
  StagedMeta *warp_meta = reinterpret_cast<StagedMeta *>(
      warp_smem + (size_t)GATHER_NBUF * (32 / TL) * a.unit_bytes);
  gather_body<TL, PACKED, CLAIM>(a, code, sruns, warp_smem, warp_meta);
}

template <int TL, int MINB, bool PACKED, bool CLAIM = false>
__global__ void __launch_bounds__(GATHER_WARPS * 32, MINB * 8 / GATHER_WARPS) gather_kernel(GatherArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ SharedRuns sruns;
  // a de-duplicated gather is launched as a dependent of the kernel clearing its table
  if (CLAIM) grid_dependency_wait();
  team_gather<TL, PACKED, CLAIM>(a, smem, sruns);
}

// Several gathers with one row geometry in one launch (e.g. one lookup batch per
// embedding table): each job has its own store, metadata, indices and output, and
// owns a contiguous range of the grid's CTAs, which run the team loop above on it.
// One launch instead of one per job removes the per-launch fixed cost (the first
// round trips of every CTA and the drain) from all jobs but one.
constexpr int BATCH_MAX_JOBS = 64;

struct BatchJob {
  const uint8_t *slots;
  int64_t slot_bytes;
  int64_t n_rows;
  const uint32_t *bitmask;
  const ibp_meta *meta;
  const int64_t *idx;
  int64_t n_idx;
  uint32_t *out;
  int cta0, ncta;
};

struct BatchArgs {
  GatherArgs common;  // geometry, status; the per-job fields are filled per CTA
  int n_jobs;
  BatchJob jobs[BATCH_MAX_JOBS];
};

template <int TL, int MINB>
__global__ void __launch_bounds__(GATHER_WARPS * 32, MINB * 8 / GATHER_WARPS)
    gather_batched_kernel(const __grid_constant__ BatchArgs b) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ SharedRuns sruns;
  int j = 0;
  while (j + 1 < b.n_jobs && (int)blockIdx.x >= b.jobs[j + 1].cta0) ++j;
  const BatchJob &job = b.jobs[j];
  GatherArgs a = b.common;
  a.slots = job.slots;
  a.slot_bytes = job.slot_bytes;
  a.n_rows = job.n_rows;
  a.bitmask = job.bitmask;
  a.meta = job.meta;
  a.idx = job.idx;
  a.n_idx = job.n_idx;
  a.out = job.out;
  a.n_units = job.n_idx * a.nseg;
  a.cta0 = job.cta0;
  a.ncta = job.ncta;
  if (a.n_units == 0) return;
  team_gather<TL, false>(a, smem, sruns);
}

// ---------------------------------------------------------------------------
// Warp-specialised variant: planner warps resolve the dependent loads, decoder
// warps stream.
//
// Planning a unit is a chain of dependent memory round trips (index -> bitmask
// bit -> header words). In the team kernel above every warp waits through that
// chain itself. Here planner warps do nothing else: one lane per unit, 32 units
// per step, each plan (source span, bit offset, participation bits, output
// position) written into a ring of plan slots in shared memory and published with
// a release arrive on the slot's "planned" mbarrier. Decoder warps run teams of TL
// lanes; a team takes its next plan (already resolved), releases the plan slot on
// its "free" mbarrier, stages the unit's bytes into its own double buffer with
// cp.async and decodes the previous unit meanwhile, so a decoder never waits on a
// dependent global load, only on its own data one unit behind.
//
// Unit k of the CTA uses plan slot k % PLAN_SLOTS. PLAN_SLOTS is a multiple of the
// CTA's decoder teams and of 32 * planners, so every use of a slot is written by the
// same planner lane and read by the same decoder team, in order: a slot's barrier is
// never more than one phase behind the unit being waited for, which the parity
// waits rely on. Every wait is bounded (mbar_wait); one that runs out records
// IBP_ERR_TIMEOUT and raises a CTA-wide abort flag that ends every loop.
// ---------------------------------------------------------------------------
constexpr int WS_PLANNERS = 2;
constexpr int WS_DECODERS = 8;
constexpr int WS_THREADS = 32 * (WS_PLANNERS + WS_DECODERS);
constexpr int PLAN_SLOTS = 512;  // measured: 4% faster than 256 on 8 KB K-cache rows

struct __align__(16) PlanSlot {
  const uint8_t *src;
  int64_t out_word;
  uint32_t nchunk, lsb, segp, nvec;
};

__device__ __forceinline__ void ws_abort(const GatherArgs &a, volatile int *abort) {
  if (!*abort) {
    report(a.status, IBP_ERR_TIMEOUT);
    *abort = 1;
  }
}

__device__ void ws_plan(const GatherArgs &a, const Code &code, int64_t u0, int64_t count,
                        int64_t r_first, PlanSlot *plans, uint64_t *planned, uint64_t *freed,
                        volatile int *abort) {
  const int lane = threadIdx.x & 31;
  const uint32_t shrink = 32u - (uint32_t)code.fc;
  const int64_t step = 32 * WS_PLANNERS;
  int64_t k = 32 * (int64_t)(threadIdx.x >> 5) + lane;
  int64_t r_next = r_first;
  for (; k - lane < count; k += step) {
    const bool have = k < count;
    int64_t r = r_next;
    r_next = k + step < count ? load_index(a, u0 + k + step, a.n_units) : -1;  // prefetch
    if (have && a.claim_table) r = claim_row(a, u0 + k, a.n_units, r);
    bool ok = true;
    if (have) {
      const Unit un = (a.offsets || a.row_bits)
                          ? plan_unit<true>(a, shrink, u0 + k, a.n_units, r, true, load_span(a, r))
                          : plan_unit<false>(a, shrink, u0 + k, a.n_units, r, true,
                                             EntrySpan{0, 0});
      const int slot = (int)(k % PLAN_SLOTS);
      ok = mbar_wait(&freed[slot], (uint32_t)((k / PLAN_SLOTS) & 1) ^ 1u, abort, a.wait_ns);
      if (ok) {
        PlanSlot p;
        p.src = un.src;
        p.out_word = un.out_word;
        p.nchunk = un.nchunk;
        p.lsb = un.lsb;
        p.segp = un.segp;
        p.nvec = un.nvec;
        plans[slot] = p;
        if (!a.withhold_plans) mbar_arrive(&planned[slot]);
      }
    }
    if (!ok) ws_abort(a, abort);
    if (__any_sync(FULL, *abort != 0)) break;
  }
}

template <int TL>
__device__ __forceinline__ Unit ws_take(const GatherArgs &a, int64_t k, int64_t count,
                                        const PlanSlot *plans, uint64_t *planned,
                                        uint64_t *freed, int tl, volatile int *abort, bool *ok) {
  Unit un;
  un.src = nullptr;
  un.out_word = 0;
  un.nchunk = 0;
  un.nvec = 0;
  un.lsb = 0;
  un.segp = 0;
  un.bmw = 0;
  un.echunk = 0;
  un.lead = 0;  // slots in device memory: spans are staged exactly
  *ok = true;
  if (k >= count) return un;
  const int slot = (int)(k % PLAN_SLOTS);
  *ok = mbar_wait(&planned[slot], (uint32_t)((k / PLAN_SLOTS) & 1), abort, a.wait_ns);
  if (*ok) {
    const PlanSlot p = plans[slot];
    un.src = p.src;
    un.out_word = p.out_word;
    un.nchunk = p.nchunk;
    un.echunk = p.nchunk;
    un.lsb = p.lsb;
    un.segp = p.segp;
    un.nvec = p.nvec;
    fetch_bitmask(a, un);
  }
  return un;
}

template <int TL>
__device__ __forceinline__ void ws_release(int64_t k, int64_t count, uint64_t *freed, int tl) {
  if (k < count && tl == 0) mbar_arrive(&freed[(int)(k % PLAN_SLOTS)]);
}

template <int NR, int TL>
__device__ void ws_decode(const GatherArgs &a, const Code &code, const SharedRuns &sruns,
                          int64_t count, const PlanSlot *plans, uint64_t *planned,
                          uint64_t *freed, uint8_t *warp_smem, volatile int *abort) {
  constexpr int TPW = 32 / TL;
  const RegRuns<NR> runs = load_runs<NR>(sruns);
  const int lane = threadIdx.x & 31;
  const int team = lane / TL;
  const int tl = lane % TL;
  const int64_t stride = (int64_t)WS_DECODERS * TPW;  // decoder teams per CTA
  const int64_t T = (int64_t)((threadIdx.x >> 5) - WS_PLANNERS) * TPW + team;
  uint8_t *const buf0 = warp_smem + team * a.unit_bytes;
  const int buf_step = TPW * a.unit_bytes;
  int64_t k = T;
  bool ok;
  Unit cur = ws_take<TL>(a, k, count, plans, planned, freed, tl, abort, &ok);
  if (!__all_sync(FULL, ok)) {
    if (lane == 0) ws_abort(a, abort);
    return;
  }
  __syncwarp();
  ws_release<TL>(k, count, freed, tl);
  stage_unit<TL>(cur, buf0, tl);
  cp_async_commit();
  int b = 0;
  for (int64_t base = T - team; base < count; base += stride) {
    const int64_t kn = k + stride;
    const Unit nxt = ws_take<TL>(a, kn, count, plans, planned, freed, tl, abort, &ok);
    if (!__all_sync(FULL, ok)) {
      if (lane == 0) ws_abort(a, abort);
      break;
    }
    __syncwarp();
    ws_release<TL>(kn, count, freed, tl);
    stage_unit<TL>(nxt, buf0 + (b ^ 1) * buf_step, tl);
    cp_async_commit();
    cp_async_wait<1>();
    __syncwarp();
    if (a.offsets || a.row_bits)
      decode_unit<NR, TL, true>(a, code, runs, sruns, cur, buf0 + b * buf_step, tl);
    else decode_unit<NR, TL, false>(a, code, runs, sruns, cur, buf0 + b * buf_step, tl);
    __syncwarp();
    cur = nxt;
    k = kn;
    b ^= 1;
  }
  cp_async_wait<0>();
}

template <int TL>
__global__ void __launch_bounds__(WS_THREADS, 2) gather_ws_kernel(GatherArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ SharedRuns sruns;
  __shared__ int abort_flag;
  __shared__ PlanSlot plans[PLAN_SLOTS];
  __shared__ uint64_t planned[PLAN_SLOTS], freed[PLAN_SLOTS];
  // a de-duplicated gather is launched as a dependent of the kernel clearing its table
  if (a.claim_table) grid_dependency_wait();
  // the CTAs split the units to gather evenly (with a device-side count, only those)
  const int64_t n_units = units_of(a);
  const int64_t u0 = n_units * blockIdx.x / gridDim.x;
  const int64_t count = n_units * (blockIdx.x + 1) / gridDim.x - u0;
  const int warp = threadIdx.x >> 5;
  // planners fetch their first indices while the metadata load is in flight
  const int64_t k_first = 32 * (int64_t)warp + (threadIdx.x & 31);
  const int64_t r_first =
      warp < WS_PLANNERS && k_first < count ? load_index(a, u0 + k_first, a.n_units) : -1;
  const ibp_meta m = load_meta(a.meta);
  if (m.dtype != a.dtype || m.block_elems != a.block_elems) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(a.status, IBP_ERR_META);
    return;
  }
  const Code code = make_code(m);
  for (int k = threadIdx.x; k < PLAN_SLOTS; k += blockDim.x) {
    mbar_init(&planned[k], 1);
    mbar_init(&freed[k], 1);
  }
  if (threadIdx.x == 0) {
    make_runs(~code.mask32, sruns);
    abort_flag = 0;
  }
  mbar_init_fence();
  __syncthreads();
  volatile int *abort = &abort_flag;
  if (warp < WS_PLANNERS) {
    ws_plan(a, code, u0, count, r_first, plans, planned, freed, abort);
    return;
  }
  uint8_t *warp_smem = smem + (size_t)(warp - WS_PLANNERS) * 2 * (32 / TL) * a.unit_bytes;
  // one decoder loop per run count: its copies are small (measured: 5% faster on
  // 2 KiB rows than one loop with the decode dispatched per unit)
  switch (sruns.n) {
    case 0: ws_decode<0, TL>(a, code, sruns, count, plans, planned, freed, warp_smem, abort); break;
    case 1: ws_decode<1, TL>(a, code, sruns, count, plans, planned, freed, warp_smem, abort); break;
    case 2: ws_decode<2, TL>(a, code, sruns, count, plans, planned, freed, warp_smem, abort); break;
    case 3: ws_decode<3, TL>(a, code, sruns, count, plans, planned, freed, warp_smem, abort); break;
    case 4: ws_decode<4, TL>(a, code, sruns, count, plans, planned, freed, warp_smem, abort); break;
    default: ws_decode<-1, TL>(a, code, sruns, count, plans, planned, freed, warp_smem, abort); break;
  }
}

int ilog2(int x) {
  int s = 0;
  while ((1 << s) < x) ++s;
  return s;
}

template <int TL, int MINB, bool PACKED, bool CLAIM = false>
int launch_tl(const GatherArgs &a, const DeviceInfo &dev, cudaStream_t s) {
  const size_t smem = (size_t)GATHER_WARPS * team_warp_bytes(TL, a.unit_bytes);
  static std::atomic<int> configured[64];  // the attribute is set once per device
  if (dev.device >= 64 || !configured[dev.device].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(gather_kernel<TL, MINB, PACKED, CLAIM>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dev.max_smem_optin - (int)sizeof(SharedRuns) - 1024) != cudaSuccess)
      return IBP_ERR_CUDA;
    if (dev.device < 64) configured[dev.device].store(1, std::memory_order_release);
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gather_kernel<TL, MINB, PACKED, CLAIM>,
                                                    GATHER_WARPS * 32, smem) != cudaSuccess ||
      per_sm < 1)
    return IBP_ERR_CUDA;
  const int64_t units_per_cta = (int64_t)GATHER_WARPS * (32 / TL);
  const int64_t want = (a.n_units + units_per_cta - 1) / units_per_cta;
  // Slots in host memory (MINB 3): the link, not the SMs, paces the gather, and 16
  // warps per SM keep it saturated (measured: within 1.5% of 24); the SM room
  // left over lets a consumer's kernels run beside a streaming decode.
  const int ctas_per_sm = MINB == 3 ? std::min(per_sm, 2 * 8 / GATHER_WARPS) : per_sm;
  const int grid = (int)std::min<int64_t>(want, (int64_t)dev.sm_count * ctas_per_sm);
  GatherArgs g = a;
  g.cta0 = 0;
  g.ncta = grid;
  if (CLAIM) {
    if (launch_dependent(gather_kernel<TL, MINB, PACKED, CLAIM>, dim3(grid),
                         dim3(GATHER_WARPS * 32), smem, s, g) != cudaSuccess)
      return IBP_ERR_CUDA;
    return IBP_OK;
  }
  gather_kernel<TL, MINB, PACKED><<<grid, GATHER_WARPS * 32, smem, s>>>(g);
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

template <int TL>
int launch_ws_tl(const GatherArgs &a, const DeviceInfo &dev, cudaStream_t s) {
  const size_t smem = (size_t)WS_DECODERS * 2 * (32 / TL) * a.unit_bytes;
  static std::atomic<int> configured[64];  // the attribute is set once per device
  if (dev.device >= 64 || !configured[dev.device].load(std::memory_order_acquire)) {
    // the largest dynamic size, leaving room for the kernel's static plan ring and
    // barriers (about 25 KB)
    if (cudaFuncSetAttribute(gather_ws_kernel<TL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dev.max_smem_optin - 28 * 1024) != cudaSuccess)
      return IBP_ERR_CUDA;
    if (dev.device < 64) configured[dev.device].store(1, std::memory_order_release);
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gather_ws_kernel<TL>, WS_THREADS,
                                                    smem) != cudaSuccess ||
      per_sm < 1)
    return IBP_ERR_CUDA;
  const int64_t want = std::max<int64_t>(1, (a.n_units + 63) / 64);
  const int grid = (int)std::min<int64_t>(want, (int64_t)dev.sm_count * per_sm);
  if (a.claim_table) {
    if (launch_dependent(gather_ws_kernel<TL>, dim3(grid), dim3(WS_THREADS), smem, s, a) !=
        cudaSuccess)
      return IBP_ERR_CUDA;
    return IBP_OK;
  }
  gather_ws_kernel<TL><<<grid, WS_THREADS, smem, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? IBP_OK : IBP_ERR_CUDA;
}

int launch_ws(GatherArgs a, const RowGeom &g, const DeviceInfo &dev, cudaStream_t s) {
  const int block_bytes = g.lwb * 4;
  a.seg_blocks = std::max(1, std::min({g.nb, 32, SEG_TARGET_BYTES / block_bytes}));
  a.nseg = (g.nb + a.seg_blocks - 1) / a.seg_blocks;
  a.unit_bytes = ((a.seg_blocks * block_bytes + 64 + 127) / 128) * 128 + 32;
  a.n_units = a.n_idx * a.nseg;
  const int nvec = a.seg_blocks * g.lwb / 4;
  int tl = 4;
  while (tl < 32 && tl * 4 < nvec) tl *= 2;
  // plan slots must be a multiple of the decoder teams and of 32 * planners
  static_assert(PLAN_SLOTS % (32 * WS_PLANNERS) == 0, "plan ring vs planners");
  static_assert(PLAN_SLOTS % (WS_DECODERS * 8) == 0, "plan ring vs decoder teams");
  switch (tl) {
    case 4: return launch_ws_tl<4>(a, dev, s);
    case 8: return launch_ws_tl<8>(a, dev, s);
    case 16: return launch_ws_tl<16>(a, dev, s);
    default: return launch_ws_tl<32>(a, dev, s);
  }
}

template <bool PACKED, bool CLAIM = false>
int launch_team(const GatherArgs &a, int tl, bool slots_in_device_memory, const DeviceInfo &dev,
                cudaStream_t s) {
  // units of at most 1 KiB in device memory: team size 4 or 8, 4 CTAs per SM (for
  // the packed and sized instantiations too: measured 10% faster than 3 on a packed
  // store in HBM).
  if (slots_in_device_memory) {
    constexpr int MINB = 4;
    if (tl == 4) return launch_tl<4, MINB, PACKED, CLAIM>(a, dev, s);
    return launch_tl<8, MINB, PACKED, CLAIM>(a, dev, s);
  }
  switch (tl) {
    case 4: return launch_tl<4, 3, PACKED, CLAIM>(a, dev, s);
    case 8: return launch_tl<8, 3, PACKED, CLAIM>(a, dev, s);
    case 16: return launch_tl<16, 3, PACKED, CLAIM>(a, dev, s);
    default: return launch_tl<32, 3, PACKED, CLAIM>(a, dev, s);
  }
}

}  // namespace

namespace {
std::atomic<uint64_t> g_wait_limit_ns{0};  // 0: WAIT_TIMEOUT_NS
std::atomic<int> g_withhold_plans{0};
}  // namespace

uint64_t gather_wait_limit_ns() {
  const uint64_t v = g_wait_limit_ns.load(std::memory_order_relaxed);
  return v ? v : WAIT_TIMEOUT_NS;
}

int gather_units_per_row(const RowGeom &g) {
  const int block_bytes = g.lwb * 4;
  const int seg_blocks = std::max(1, std::min({g.nb, 32, SEG_TARGET_BYTES / block_bytes}));
  return (g.nb + seg_blocks - 1) / seg_blocks;
}

int launch_gather(const void *slots, int64_t slot_bytes, const uint64_t *d_offsets,
                  uint64_t packed_bytes, int64_t n_rows, const RowGeom &g, uint32_t dtype,
                  const uint32_t *d_bitmask, const ibp_meta *d_meta, const int64_t *d_idx,
                  int64_t row0, int64_t n_idx, void *out, int32_t *d_status,
                  bool slots_in_device_memory, cudaStream_t s, const uint32_t *d_row_bits,
                  bool skip_negative, bool pos_in_index,
                  const unsigned long long *d_idx_count, const ClaimTable *claim) {
  if (n_idx == 0) return IBP_OK;
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  GatherArgs a;
  a.slots = static_cast<const uint8_t *>(slots);
  a.slot_bytes = slot_bytes;
  a.cta0 = 0;
  a.ncta = 0;
  a.offsets = d_offsets;
  a.row_bits = d_offsets ? nullptr : d_row_bits;
  a.span_align = slots_in_device_memory ? 16u : 128u;
  a.skip_negative = skip_negative ? 1u : 0u;
  a.pos_in_index = pos_in_index ? 1u : 0u;
  a.idx_count = d_idx_count;
  a.wait_ns = gather_wait_limit_ns();
  a.withhold_plans = g_withhold_plans.load(std::memory_order_relaxed) ? 1u : 0u;
  a.claim_table = claim ? claim->table : nullptr;
  a.claim_mask = claim ? claim->mask : 0u;
  a.claim_owner = claim ? claim->owner : nullptr;
  if (claim && (d_offsets || d_row_bits || gather_units_per_row(g) != 1)) return IBP_ERR_ARG;
  a.packed_bytes = d_offsets ? packed_bytes : (uint64_t)n_rows * (uint64_t)slot_bytes;
  a.n_rows = n_rows;
  a.bitmask = d_bitmask;
  a.meta = d_meta;
  a.idx = d_idx;
  a.row0 = row0;
  a.n_idx = n_idx;
  a.out = static_cast<uint32_t *>(out);
  a.status = d_status;
  a.dtype = dtype;
  a.block_elems = (uint32_t)g.B;
  a.lwb = g.lwb;
  a.lwb_shift = ilog2(g.lwb);
  a.nb = g.nb;
  a.raw_words = g.raw_words;
  a.lwt = g.lwt;
  a.raw_bytes = g.raw_bytes;
  // Slots in device memory with units of more than 1 KiB: the warp-specialised
  // kernel (planning off the decoders' path pays once a unit takes several vectors
  // per lane). Small units, and slots in host memory, which the link paces: the
  // team kernel (every warp decodes; measured faster there).
  const int block_bytes_all = g.lwb * 4;
  const int unit_raw = std::max(1, std::min({g.nb, 32, SEG_TARGET_BYTES / block_bytes_all})) *
                       block_bytes_all;
  if (slots_in_device_memory && unit_raw > 1024) return launch_ws(a, g, dev, s);
  const int block_bytes = g.lwb * 4;
  a.seg_blocks = std::max(1, std::min({g.nb, 32, SEG_TARGET_BYTES / block_bytes}));
  a.nseg = (g.nb + a.seg_blocks - 1) / a.seg_blocks;
  // staged bytes <= segment raw bytes + 32 (alignment), + 8 for the word after the
  // last field; padded so that the teams' buffers start 8 banks apart
  a.unit_bytes = ((a.seg_blocks * block_bytes + 64 + 127) / 128) * 128 + 32;
  a.n_units = n_idx * a.nseg;
  // team size: about four 16-byte vectors per lane
  const int nvec = a.seg_blocks * g.lwb / 4;
  int tl = 4;
  while (tl < 32 && tl * 4 < nvec) tl *= 2;
  if (d_offsets || a.row_bits) return launch_team<true>(a, tl, slots_in_device_memory, dev, s);
  if (a.claim_table) return launch_team<false, true>(a, tl, slots_in_device_memory, dev, s);
  return launch_team<false>(a, tl, slots_in_device_memory, dev, s);
}

int launch_gather_batched(const ibp_gather_job *jobs, int n_jobs, const RowGeom &g,
                          uint32_t dtype, int32_t *d_status, const bool *in_device,
                          cudaStream_t s) {
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  BatchArgs b;
  GatherArgs &a = b.common;
  a = GatherArgs{};
  a.span_align = 16u;
  a.skip_negative = 0u;
  a.pos_in_index = 0u;
  a.idx_count = nullptr;
  a.wait_ns = gather_wait_limit_ns();
  a.status = d_status;
  a.dtype = dtype;
  a.block_elems = (uint32_t)g.B;
  a.lwb = g.lwb;
  a.lwb_shift = ilog2(g.lwb);
  a.nb = g.nb;
  a.raw_words = g.raw_words;
  a.lwt = g.lwt;
  a.raw_bytes = g.raw_bytes;
  const int block_bytes = g.lwb * 4;
  a.seg_blocks = std::max(1, std::min({g.nb, 32, SEG_TARGET_BYTES / block_bytes}));
  a.nseg = (g.nb + a.seg_blocks - 1) / a.seg_blocks;
  a.unit_bytes = ((a.seg_blocks * block_bytes + 64 + 127) / 128) * 128 + 32;
  const int nvec = a.seg_blocks * g.lwb / 4;
  int tl = 4;
  while (tl < 32 && tl * 4 < nvec) tl *= 2;
  for (int j0 = 0; j0 < n_jobs; j0 += BATCH_MAX_JOBS) {
    const int nj = std::min(BATCH_MAX_JOBS, n_jobs - j0);
    bool all_device = true;
    int64_t total_units = 0;
    for (int j = 0; j < nj; ++j) {
      all_device = all_device && in_device[j0 + j];
      total_units += jobs[j0 + j].n_idx * a.nseg;
    }
    if (total_units == 0) continue;
    const int minb = all_device ? 4 : 3;
    // CTAs in proportion to each job's units, at least one per job with work
    int per_sm = 0;
    const size_t smem = (size_t)GATHER_WARPS * team_warp_bytes(tl, a.unit_bytes);
    const void *kern = nullptr;
#define IBP_BATCH_KERNEL(T, M) reinterpret_cast<const void *>(gather_batched_kernel<T, M>)
    switch (tl) {
      case 4: kern = minb == 4 ? IBP_BATCH_KERNEL(4, 4) : IBP_BATCH_KERNEL(4, 3); break;
      case 8: kern = minb == 4 ? IBP_BATCH_KERNEL(8, 4) : IBP_BATCH_KERNEL(8, 3); break;
      case 16: kern = minb == 4 ? IBP_BATCH_KERNEL(16, 4) : IBP_BATCH_KERNEL(16, 3); break;
      default: kern = minb == 4 ? IBP_BATCH_KERNEL(32, 4) : IBP_BATCH_KERNEL(32, 3); break;
    }
#undef IBP_BATCH_KERNEL
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dev.max_smem_optin - (int)sizeof(SharedRuns) - 1024) != cudaSuccess)
      return IBP_ERR_CUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, GATHER_WARPS * 32, smem) !=
            cudaSuccess ||
        per_sm < 1)
      return IBP_ERR_CUDA;
    const int ctas_per_sm = minb == 3 ? std::min(per_sm, 2) : per_sm;
    const int64_t budget = (int64_t)dev.sm_count * ctas_per_sm;
    const int64_t units_per_cta = (int64_t)GATHER_WARPS * (32 / tl);
    int cta = 0;
    int used = 0;
    for (int j = 0; j < nj; ++j) {
      const ibp_gather_job &src = jobs[j0 + j];
      const int64_t units = src.n_idx * a.nseg;
      int64_t n = 0;
      if (units > 0) {
        const int64_t want = (units + units_per_cta - 1) / units_per_cta;
        const int64_t share = std::max<int64_t>(1, budget * units / total_units);
        n = std::min(want, share);
      }
      BatchJob &d = b.jobs[used];
      if (units == 0) continue;
      d.slots = static_cast<const uint8_t *>(src.slots);
      d.slot_bytes = src.slot_bytes;
      d.n_rows = src.n_rows;
      d.bitmask = src.d_row_bitmask;
      d.meta = src.d_meta;
      d.idx = src.d_idx;
      d.n_idx = src.n_idx;
      d.out = static_cast<uint32_t *>(src.out);
      d.cta0 = cta;
      d.ncta = (int)n;
      cta += (int)n;
      ++used;
    }
    b.n_jobs = used;
    switch (tl) {
      case 4:
        if (minb == 4) gather_batched_kernel<4, 4><<<cta, GATHER_WARPS * 32, smem, s>>>(b);
        else gather_batched_kernel<4, 3><<<cta, GATHER_WARPS * 32, smem, s>>>(b);
        break;
      case 8:
        if (minb == 4) gather_batched_kernel<8, 4><<<cta, GATHER_WARPS * 32, smem, s>>>(b);
        else gather_batched_kernel<8, 3><<<cta, GATHER_WARPS * 32, smem, s>>>(b);
        break;
      case 16:
        if (minb == 4) gather_batched_kernel<16, 4><<<cta, GATHER_WARPS * 32, smem, s>>>(b);
        else gather_batched_kernel<16, 3><<<cta, GATHER_WARPS * 32, smem, s>>>(b);
        break;
      default:
        if (minb == 4) gather_batched_kernel<32, 4><<<cta, GATHER_WARPS * 32, smem, s>>>(b);
        else gather_batched_kernel<32, 3><<<cta, GATHER_WARPS * 32, smem, s>>>(b);
        break;
    }
    if (cudaGetLastError() != cudaSuccess) return IBP_ERR_CUDA;
  }
  return IBP_OK;
}

}  // namespace ibp

extern "C" uint64_t ibp_testing_set_wait_limit_ns(uint64_t ns) {
  return ibp::g_wait_limit_ns.exchange(ns, std::memory_order_relaxed);
}

extern "C" int ibp_testing_withhold_plans(int on) {
  return ibp::g_withhold_plans.exchange(on ? 1 : 0, std::memory_order_relaxed);
}
