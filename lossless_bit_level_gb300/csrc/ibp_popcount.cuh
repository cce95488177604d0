// Bit-sliced positional population count (Harley-Seal carry-save adders), shared by
// the metadata kernels: P.tot[j] (after flush_eights and the final fold) counts the
// added words whose bit j is 1.
#pragma once

#include <stdint.h>

namespace ibp {

__device__ __forceinline__ void csa(uint32_t &h, uint32_t &l, uint32_t a, uint32_t b, uint32_t c) {
  const uint32_t u = a ^ b;
  h = (a & b) | (u & c);
  l = u ^ c;
}

struct Planes {
  uint32_t ones = 0, twos = 0, fours = 0;
  uint32_t eights[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // ripple counter of eights, bit-sliced
  uint32_t tot[32];
};

__device__ __forceinline__ void add8(Planes &P, const uint4 &a, const uint4 &b) {
  uint32_t twosA, twosB, foursA, foursB, eights;
  csa(twosA, P.ones, P.ones, a.x, a.y);
  csa(twosB, P.ones, P.ones, a.z, a.w);
  csa(foursA, P.twos, P.twos, twosA, twosB);
  csa(twosA, P.ones, P.ones, b.x, b.y);
  csa(twosB, P.ones, P.ones, b.z, b.w);
  csa(foursB, P.twos, P.twos, twosA, twosB);
  csa(eights, P.fours, P.fours, foursA, foursB);
  uint32_t carry = eights;
#pragma unroll
  for (int l = 0; l < 8; ++l) {
    const uint32_t t = P.eights[l] & carry;
    P.eights[l] ^= carry;
    carry = t;
  }
}

__device__ __forceinline__ void flush_eights(Planes &P) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    uint32_t c = 0;
#pragma unroll
    for (int l = 0; l < 8; ++l) c |= ((P.eights[l] >> j) & 1u) << l;
    P.tot[j] += 8u * c;
  }
#pragma unroll
  for (int l = 0; l < 8; ++l) P.eights[l] = 0;
}

// Fold the remaining ones/twos/fours planes into the totals (after a flush).
__device__ __forceinline__ void fold_planes(Planes &P) {
#pragma unroll
  for (int j = 0; j < 32; ++j)
    P.tot[j] += ((P.ones >> j) & 1u) + 2u * ((P.twos >> j) & 1u) + 4u * ((P.fours >> j) & 1u);
}

}  // namespace ibp
