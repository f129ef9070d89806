// Philox4x32-10 counter-based generator (Salmon, Moraes, Dror, Shaw, "Parallel
// random numbers: as easy as 1, 2, 3", SC 2011), for dropout.
//
// One call maps a 128-bit counter (x0, x1, x2, x3) and a 64-bit key (k0, k1)
// to four 32-bit words by ten rounds of
//   hi0:lo0 = M0 * x0, hi1:lo1 = M1 * x2  (32 x 32 -> 64-bit products)
//   (x0, x1, x2, x3) <- (hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0)
// with the key bumped by the Weyl increments (W0, W1) between rounds. The
// multipliers and increments are the paper's constants for Philox4x32.
#pragma once
#include <stdint.h>

namespace fa {

struct Philox4 {
  uint32_t v[4];
};

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3, uint32_t k0,
                                                  uint32_t k1) {
  constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  constexpr uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(M0, x0), lo0 = M0 * x0;
    const uint32_t hi1 = __umulhi(M1, x2), lo1 = M1 * x2;
    const uint32_t y0 = hi1 ^ x1 ^ k0, y2 = hi0 ^ x3 ^ k1;
    x0 = y0;
    x1 = lo1;
    x2 = y2;
    x3 = lo0;
    k0 += W0;
    k1 += W1;
  }
  return Philox4{{x0, x1, x2, x3}};
}

// Dropout of attention probabilities (page "FlashAttention：快速且内存高效的准确注意力机制",
// section "参数说明": dropout_p; the pages give no generator). Element (b, h, i, j)
// of the (per-sequence) probability matrix uses word j % 4 of
//   philox4x32_10(counter = (j / 4, i, b * H + h, offset), key = (seed_lo, seed_hi))
// and is dropped when that word is below thr = floor(p * 2^32); kept entries
// are scaled by 1 / (1 - p).
struct Dropout {
  uint32_t thr;      // 0: no dropout
  float keep_scale;  // 1 / (1 - p)
  uint32_t seed_lo, seed_hi, offset;
};

// The four keep flags of key group j4 = j / 4 for row i of head bh (bit e: key 4 * j4 + e kept).
__device__ __forceinline__ uint32_t dropout_keep4(const Dropout& d, int bh, int i, int j4) {
  const Philox4 r = philox4x32_10(uint32_t(j4), uint32_t(i), uint32_t(bh), d.offset, d.seed_lo, d.seed_hi);
  return uint32_t(r.v[0] >= d.thr) | (uint32_t(r.v[1] >= d.thr) << 1) | (uint32_t(r.v[2] >= d.thr) << 2) |
         (uint32_t(r.v[3] >= d.thr) << 3);
}

}  // namespace fa
