// Rotary position embedding of one 16-byte chunk (8 elements) of a head row.
//
// Page "FlashAttention：快速且内存高效的准确注意力机制", section "2.2：针对推理进行优化":
// flash_attn_with_kvcache applies rotary embeddings. The pages give no formula;
// the standard rotary embedding is taken, with the caller's cos/sin tables
// (rot_len, rot_dim / 2): the pair (x1, x2) at frequency f and position pos
// becomes (x1 cos - x2 sin, x1 sin + x2 cos), cos = cos_tab[pos][f]. Pairs are
// (2f, 2f + 1) when interleaved, else (f, f + rot_dim / 2); elements at or
// beyond rot_dim are unchanged. rot_dim is a multiple of 16, so a chunk lies
// wholly inside or outside the rotated dims and a half-split partner is the
// chunk rot_dim / 2 elements away.
#pragma once
#include <stdint.h>

namespace fa {

struct Rotary {
  const float* cos;  // (len, dim / 2), fp32; NULL: no rotation
  const float* sin;
  int dim, len, interleaved;
};

// x: this chunk (elements d0 .. d0 + 7), partner: the chunk at d0 -/+ dim/2
// (read only when not interleaved). pos is clamped to [0, len - 1].
__device__ __forceinline__ void rotary8(float (&x)[8], const float (&partner)[8], int d0, int pos, const Rotary& r) {
  if (r.cos == nullptr || d0 >= r.dim) return;
  pos = pos < 0 ? 0 : (pos >= r.len ? r.len - 1 : pos);
  const float* ct = r.cos + size_t(pos) * (r.dim / 2);
  const float* st = r.sin + size_t(pos) * (r.dim / 2);
  if (r.interleaved) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int f = d0 / 2 + e;
      const float c = ct[f], s = st[f], x1 = x[2 * e], x2 = x[2 * e + 1];
      x[2 * e] = x1 * c - x2 * s;
      x[2 * e + 1] = x1 * s + x2 * c;
    }
  } else {
    const int half = r.dim / 2;
    const bool first = d0 < half;  // this chunk holds x1 of its pairs, the partner x2
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int f = (first ? d0 : d0 - half) + e;
      const float c = ct[f], s = st[f];
      x[e] = first ? (x[e] * c - partner[e] * s) : (partner[e] * s + x[e] * c);
    }
  }
}

// Element offset of the partner chunk of the chunk starting at d0 (half-split pairs).
__device__ __forceinline__ int rotary_partner(int d0, const Rotary& r) {
  return d0 < r.dim / 2 ? d0 + r.dim / 2 : d0 - r.dim / 2;
}

}  // namespace fa
