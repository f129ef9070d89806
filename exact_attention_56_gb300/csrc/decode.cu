// Split-KV decode for short queries, plus the merge kernel.
//
// Page "FlashAttention：快速且内存高效的准确注意力机制", section
// "2.2：针对推理进行优化": with a very short query the cost is reading the KV
// cache; the key range is cut into splits handled by separate thread blocks,
// and a separate kernel merges the per-split results.
//
// Split kernel (one CTA per (split, key/value head, batch, block of R query
// pairs)): the Sq x group (query row, query head) pairs that read one key/value
// head are served R at a time, so each K/V tile is read once for all of them
// rather than once per query head and row. The caches are dense (B, Sk, Hk, D)
// or pages addressed through a block table:
//   warp 4      TMA producer: streams 32 KB stages (TK keys of K and of V,
//               128-byte swizzled) through an mbarrier ring.
//   warps 0..3  consumers: thread (g, c) owns 16-byte chunk c of the head dim
//               and key lane g; a group of D/8 lanes shares one key at a time
//               (dot products reduced with shuffles), keeps its own online
//               softmax state (m, l) and its 8 output columns per query pair,
//               and the groups are merged once at the end through shared memory.
//   Output: per split the normalised partial O_s (fp32, D) and L_s (natural
//   log) in the workspace; a split with no live key writes O_s = 0, L_s = -inf.
// Merge kernel (one warp per (batch, query row, head)):
//   L = log sum_s exp(L_s), O = sum_s exp(L_s - L) O_s, vectorised 16-byte loads.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "../../include/fa.h"
#include "internal.h"
#include "ptx.cuh"
#include "rotary.cuh"

namespace fa {

template <int D>
struct DecCfg {
  static constexpr int CH = D / 8;               // 16-byte chunks per row
  static constexpr int G = 128 / CH;             // key lanes among the 128 consumer threads
  static constexpr int KPL = 8;                  // keys per lane per tile
  static constexpr int TK = G * KPL;             // keys per tile
  static constexpr int PANELS = D / 64;
  static constexpr int PANEL_BYTES = TK * 128;   // TK rows x 128 B
  static constexpr int TILE_BYTES = PANELS * PANEL_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile then V tile
  static constexpr int NSTAGE = 3;
  static constexpr int THREADS = 160;            // 4 consumer warps + 1 producer warp
  static constexpr int RED_OFF = NSTAGE * STAGE_BYTES;
  static constexpr int RED_BYTES = G * D * 4 + 2 * G * 4;
  static constexpr int BAR_OFF = RED_OFF + RED_BYTES;
  static constexpr int SMEM_BYTES = BAR_OFF + 128 + 1024;
  static_assert(STAGE_BYTES == 32768, "stage size");
};

struct DecParams {
  const __nv_bfloat16* q;
  float* part_o;  // [B][Sq][H][n][D]
  float* part_l;  // [B][Sq][H][n]
  const float* alibi;
  int alibi_bstride;
  int B, Sq, Sk, H, n_splits;  // Sk: with a page table, the longest sequence
  int group;  // query heads per key/value head (H / Hk)
  int n_rb;   // CTAs (row blocks) per key/value head: ceil(Sq * group / R)
  // Paged KV cache (page section "2.5：分页KV缓存"): NULL for the dense
  // (B, Sk, Hk, D) caches; else logical key block p of sequence b lives in page
  // block_table[b * max_pages + p] of (num_pages, page_size, Hk, D) caches and
  // the sequence has seqlens_k[b] keys. page_size is a multiple of TK.
  const int* block_table;
  const int* seqlens_k;
  int page_size, max_pages;
  // With seqlens_k, sequence b has min(seqlens_k[b] + s_new, cap) keys: s_new
  // rows appended in this call behind seqlens_k[b] cached ones, cap the rows the
  // cache holds per sequence.
  int s_new, cap;
  Rotary rot;  // rotation of q, row i at position i + Sk_b - Sq (rot.cos NULL: none)
  int wl, wr;
  float scale_log2;
  unsigned int* status;
};

struct DecBars {
  uint64_t full[4];
  uint64_t empty[4];
  int abort;
};

enum : uint32_t { SITE_DEC_EMPTY = 0x21, SITE_DEC_FULL = 0x22 };

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = __uint_as_float(w[e] << 16);
    f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <int D, int R>
__global__ void __launch_bounds__(DecCfg<D>::THREADS)
    fa_decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                           const DecParams p) {
  using C = DecCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  DecBars* bars = reinterpret_cast<DecBars*>(smem + C::BAR_OFF);
  float* red_o = reinterpret_cast<float*>(smem + C::RED_OFF);  // [G][D]
  float* red_m = red_o + C::G * D;                               // [G]
  float* red_l = red_m + C::G;                                   // [G]

  // This CTA serves up to R of the Sq x group (query row, query head) pairs
  // that read key/value head hk; every K/V tile it loads is used by all of them.
  const int split = blockIdx.x;
  const int hk = blockIdx.y / p.n_rb;
  const int rb = blockIdx.y % p.n_rb;
  const int b = blockIdx.z;
  const int n_pairs = p.Sq * p.group;
  // this sequence's keys, clamped to what the cache (or its page table) holds
  const int Sk = p.seqlens_k ? max(0, min(p.seqlens_k[b] + p.s_new, p.cap)) : p.Sk;
  // Splits cut the key range at whole tiles, so a tile never straddles a page.
  // Row k sees keys [klo[k], khi[k]): its live range clipped to this split; the
  // CTA streams the tiles covering the union of those ranges.
  const int n_all = (Sk + C::TK - 1) / C::TK;
  const int s_lo = int((long long)n_all * split / p.n_splits) * C::TK;
  const int s_hi = min(Sk, int((long long)n_all * (split + 1) / p.n_splits) * C::TK);  // exclusive
  int ri[R], rh[R], klo[R], khi[R];
  int ks = Sk, ke = 0;
#pragma unroll
  for (int k = 0; k < R; ++k) {
    const int r = rb * R + k;
    ri[k] = r / p.group;                  // query row
    rh[k] = hk * p.group + r % p.group;   // query head
    klo[k] = 1;
    khi[k] = 0;
    if (r < n_pairs) {
      const RowRange rr = live_range(ri[k], p.Sq, Sk, p.wl, p.wr);
      klo[k] = max(s_lo, rr.lo);
      khi[k] = min(s_hi, rr.hi + 1);
      if (khi[k] > klo[k]) {
        ks = min(ks, klo[k]);
        ke = max(ke, khi[k]);
      }
    }
  }
  const int t0 = (ks / C::TK) * C::TK;  // first tile, aligned
  const int n_tiles = ke > ks ? (ke - t0 + C::TK - 1) / C::TK : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 128);
    }
    bars->abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const Watch watch{&bars->abort, p.status};

  if (threadIdx.x >= 128) {
    // ------------------------------------------------------------ producer
    if (threadIdx.x == 128 && n_tiles > 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int issued = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % C::NSTAGE;
        const uint32_t ph = uint32_t(t / C::NSTAGE) & 1u;
        if (!fa_wait(&bars->empty[s], ph ^ 1u, watch, SITE_DEC_EMPTY)) break;
        uint8_t* st = smem + s * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&bars->full[s], C::STAGE_BYTES);
        int row = t0 + t * C::TK, tb = b;
        if (p.block_table) {  // (row in page, page) coordinates of this tile
          tb = p.block_table[size_t(b) * p.max_pages + row / p.page_size];
          row %= p.page_size;
        }
#pragma unroll
        for (int pn = 0; pn < C::PANELS; ++pn) {
          tma_load_4d(st + pn * C::PANEL_BYTES, &tm_k, &bars->full[s], pn * 64, hk, row, tb);
          tma_load_4d(st + C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_v, &bars->full[s], pn * 64, hk, row, tb);
        }
        issued = t + 1;
      }
      // Every copy must have landed before this CTA may exit (consumers that
      // aborted early no longer wait for them).
      {
        for (int t = (issued > C::NSTAGE ? issued - C::NSTAGE : 0); t < issued; ++t) {
          const uint32_t a = smem_u32(&bars->full[t % C::NSTAGE]);
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(a, uint32_t(t / C::NSTAGE) & 1u))
            if (globaltimer_ns() - t0 > FA_WAIT_TIMEOUT_NS) break;
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int tid = threadIdx.x;
  const int c = tid % C::CH;
  const int g = tid / C::CH;
  const bool has_alibi = p.alibi != nullptr;
  float qf[R][8], slope_log2[R];
  int c_i[R];
#pragma unroll
  for (int k = 0; k < R; ++k) {
    c_i[k] = ri[k] + Sk - p.Sq;
    slope_log2[k] = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) qf[k][e] = 0.0f;
    if (khi[k] <= klo[k]) continue;  // no live key in this split (or no such pair)
    const __nv_bfloat16* qrow = p.q + ((size_t(b) * p.Sq + ri[k]) * p.H + rh[k]) * D;
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(qrow + c * 8), qf[k]);
    if (p.rot.cos != nullptr && c * 8 < p.rot.dim) {  // rotary at the row's diagonal position
      float pq[8];
      if (!p.rot.interleaved)
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(qrow + rotary_partner(c * 8, p.rot)), pq);
      rotary8(qf[k], pq, c * 8, c_i[k], p.rot);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) qf[k][e] *= p.scale_log2;
    if (has_alibi) slope_log2[k] = p.alibi[b * p.alibi_bstride + rh[k]] * 1.4426950408889634f;
  }
  const int pn = c / 8;
  const int cc = c % 8;

  float m[R], l[R], o[R][8];
#pragma unroll
  for (int k = 0; k < R; ++k) {
    m[k] = -INFINITY;
    l[k] = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[k][e] = 0.0f;
  }

  for (int t = 0; t < n_tiles; ++t) {
    const int s = t % C::NSTAGE;
    if (!fa_wait_warp(&bars->full[s], uint32_t(t / C::NSTAGE) & 1u, watch, SITE_DEC_FULL)) break;
    const uint8_t* kt = smem + s * C::STAGE_BYTES + pn * C::PANEL_BYTES;
    const uint8_t* vt = kt + C::TILE_BYTES;
    const int row0 = t0 + t * C::TK;
    float sc[R][C::KPL];
#pragma unroll
    for (int u = 0; u < C::KPL; ++u) {
      const int kr = g + C::G * u;
      const uint4 kv = *reinterpret_cast<const uint4*>(kt + kr * 128 + ((cc ^ (kr & 7)) << 4));
      float kf[8];
      bf16x8_to_f32(kv, kf);
      const int kj = row0 + kr;
#pragma unroll
      for (int k = 0; k < R; ++k) {
        float d = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) d = fmaf(qf[k][e], kf[e], d);
#pragma unroll
        for (int off = C::CH / 2; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
        if (has_alibi) d -= slope_log2[k] * fabsf(float(c_i[k] - kj));
        sc[k][u] = (kj >= klo[k] && kj < khi[k]) ? d : -INFINITY;
      }
    }
    float m_use[R];
#pragma unroll
    for (int k = 0; k < R; ++k) {
      float mt = sc[k][0];
#pragma unroll
      for (int u = 1; u < C::KPL; ++u) mt = fmaxf(mt, sc[k][u]);
      const float m_new = fmaxf(m[k], mt);
      if (m_new != -INFINITY) {
        if (m[k] == -INFINITY) {
          m[k] = m_new;
        } else if (m_new > m[k] + 8.0f) {
          const float alpha = ex2_approx(m[k] - m_new);
          l[k] *= alpha;
#pragma unroll
          for (int e = 0; e < 8; ++e) o[k][e] *= alpha;
          m[k] = m_new;
        }
      }
      m_use[k] = (m[k] == -INFINITY) ? 0.0f : m[k];
    }
#pragma unroll
    for (int u = 0; u < C::KPL; ++u) {
      const int kr = g + C::G * u;
      const uint4 vv = *reinterpret_cast<const uint4*>(vt + kr * 128 + ((cc ^ (kr & 7)) << 4));
      float vf[8];
      bf16x8_to_f32(vv, vf);
#pragma unroll
      for (int k = 0; k < R; ++k) {
        const float pu = ex2_approx(sc[k][u] - m_use[k]);
        l[k] += pu;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[k][e] = fmaf(pu, vf[e], o[k][e]);
      }
    }
    mbar_arrive(&bars->empty[s]);
  }

  // Merge the G key lanes of this CTA, one row at a time through shared memory.
#pragma unroll
  for (int k = 0; k < R; ++k) {
    const int r = rb * R + k;
    if (c == 0) {
      red_m[g] = m[k];
      red_l[g] = l[k];
    }
    named_bar_sync(1, 128);
    float M = -INFINITY;
#pragma unroll
    for (int gg = 0; gg < C::G; ++gg) M = fmaxf(M, red_m[gg]);
    const float Ms = (M == -INFINITY) ? 0.0f : M;
    const float wg = (m[k] == -INFINITY) ? 0.0f : ex2_approx(m[k] - Ms);
#pragma unroll
    for (int e = 0; e < 8; ++e) red_o[g * D + c * 8 + e] = o[k][e] * wg;
    named_bar_sync(1, 128);
    if (r < n_pairs) {  // a split with no live key for this row writes O_s = 0, L_s = -inf
      float L = 0.0f;
#pragma unroll
      for (int gg = 0; gg < C::G; ++gg)
        L += (red_m[gg] == -INFINITY) ? 0.0f : red_l[gg] * ex2_approx(red_m[gg] - Ms);
      const float inv = L > 0.0f ? 1.0f / L : 0.0f;
      const size_t pidx = ((size_t(b) * p.Sq + ri[k]) * p.H + rh[k]) * p.n_splits + split;
      for (int d = tid; d < D; d += 128) {
        float acc = 0.0f;
#pragma unroll
        for (int gg = 0; gg < C::G; ++gg) acc += red_o[gg * D + d];
        p.part_o[pidx * D + d] = acc * inv;
      }
      if (tid == 0) p.part_l[pidx] = L > 0.0f ? (M + lg2_approx(L)) * 0.6931471805599453f : -INFINITY;
    }
    named_bar_sync(1, 128);  // red_* are reused by the next row
  }
}

// Appends s_new rows of k_new, v_new (B, s_new, Hk, D) to the cache at
// positions seqlens[b] + s, the keys rotated at their positions (page section
// "2.2": flash_attn_with_kvcache updates the KV cache in place and applies
// rotary embeddings). One thread per 16-byte chunk; rows past the cache's
// capacity, and rows whose page index lies outside the cache, are not written.
template <int D>
__global__ void __launch_bounds__(256) fa_kv_append_kernel(const __nv_bfloat16* __restrict__ k_new,
                                                           const __nv_bfloat16* __restrict__ v_new,
                                                           __nv_bfloat16* k_cache, __nv_bfloat16* v_cache,
                                                           const int* seqlens, const int* block_table, int B,
                                                           int s_new, int Hk, int cap, int num_pages, int page_size,
                                                           int max_pages, Rotary rot) {
  constexpr int CPR = D / 8;
  const long long n = (long long)B * s_new * Hk * CPR;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < n;
       it += (long long)gridDim.x * blockDim.x) {
    const int c = int(it % CPR);
    const long long row = it / CPR;  // (b * s_new + s) * Hk + hk
    const int hk = int(row % Hk);
    const int s = int((row / Hk) % s_new);
    const int b = int(row / (Hk * (long long)s_new));
    const int pos = seqlens[b] + s;
    if (pos < 0 || pos >= cap) continue;
    size_t dst_row;
    if (block_table) {
      const int page = block_table[size_t(b) * max_pages + pos / page_size];
      if (page < 0 || page >= num_pages) continue;
      dst_row = size_t(page) * page_size + pos % page_size;
    } else {
      dst_row = size_t(b) * cap + pos;
    }
    const size_t src = size_t(row) * D;
    const size_t dst = (dst_row * Hk + hk) * D + c * 8;
    *reinterpret_cast<uint4*>(v_cache + dst) = *reinterpret_cast<const uint4*>(v_new + src + c * 8);
    uint4 kv = *reinterpret_cast<const uint4*>(k_new + src + c * 8);
    if (rot.cos != nullptr && c * 8 < rot.dim) {
      float x[8], px[8];
      bf16x8_to_f32(kv, x);
      if (!rot.interleaved) bf16x8_to_f32(*reinterpret_cast<const uint4*>(k_new + src + rotary_partner(c * 8, rot)), px);
      rotary8(x, px, c * 8, pos, rot);
      kv = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                      pack_bf16x2(x[6], x[7]));
    }
    *reinterpret_cast<uint4*>(k_cache + dst) = kv;
  }
}

// One warp per (b, query row, head).
template <int D>
__global__ void __launch_bounds__(256) fa_decode_combine_kernel(const float* __restrict__ part_o,
                                                                 const float* __restrict__ part_l,
                                                                 __nv_bfloat16* __restrict__ out,
                                                                 float* __restrict__ lse, int B, int Sq, int H,
                                                                 int n) {
  constexpr int PER = D / 32;  // columns per lane: 2, 4 or 8
  const int warp_global = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (warp_global >= B * Sq * H) return;
  const int h = warp_global % H;
  const int i = (warp_global / H) % Sq;
  const int b = warp_global / (H * Sq);
  const size_t base = size_t(warp_global) * n;
  float M = -INFINITY;
  for (int s = lane; s < n; s += 32) M = fmaxf(M, part_l[base + s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float Ms = (M == -INFINITY) ? 0.0f : M;
  float Z = 0.0f;
  for (int s = lane; s < n; s += 32) {
    const float ls = part_l[base + s];
    Z += (ls == -INFINITY) ? 0.0f : __expf(ls - Ms);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, off);
  const float invZ = Z > 0.0f ? 1.0f / Z : 0.0f;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.0f;
  for (int s = 0; s < n; ++s) {
    const float ls = part_l[base + s];
    if (ls == -INFINITY) continue;
    const float w = __expf(ls - Ms) * invZ;
    const float* src = part_o + (base + s) * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; e += 2) {
      const float2 v2 = *reinterpret_cast<const float2*>(src + e);
      acc[e] = fmaf(w, v2.x, acc[e]);
      acc[e + 1] = fmaf(w, v2.y, acc[e + 1]);
    }
  }
  uint32_t pk[PER / 2];
#pragma unroll
  for (int e = 0; e < PER / 2; ++e) pk[e] = pack_bf16x2(acc[2 * e], acc[2 * e + 1]);
  __nv_bfloat16* dst = out + ((size_t(b) * Sq + i) * H + h) * D + lane * PER;
  if constexpr (PER == 2) {
    *reinterpret_cast<uint32_t*>(dst) = pk[0];
  } else if constexpr (PER == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(pk[0], pk[1]);
  } else {
    *reinterpret_cast<uint4*>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
  if (lane == 0) lse[(size_t(b) * H + h) * Sq + i] = (Z > 0.0f) ? Ms + __logf(Z) : -INFINITY;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int kv_append_launch(const AttnShape& s, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                     const CacheArgs& c, cudaStream_t stream) {
  if (c.s_new < 1) return FA_OK;
  const long long items = (long long)s.B * c.s_new * s.Hk * (s.D / 8);
  const long long cap_blocks = (long long)device_sm_count() * 8;
  const int grid = int(std::max(1LL, std::min(cap_blocks, (items + 255) / 256)));
  const auto* kn = static_cast<const __nv_bfloat16*>(k_new);
  const auto* vn = static_cast<const __nv_bfloat16*>(v_new);
  auto* kc = static_cast<__nv_bfloat16*>(k_cache);
  auto* vc = static_cast<__nv_bfloat16*>(v_cache);
  switch (s.D) {
    case 64:
      fa_kv_append_kernel<64><<<grid, 256, 0, stream>>>(kn, vn, kc, vc, c.seqlens, c.block_table, s.B, c.s_new, s.Hk,
                                                          c.cap, c.num_pages, c.page_size, c.max_pages, c.rot);
      break;
    case 128:
      fa_kv_append_kernel<128><<<grid, 256, 0, stream>>>(kn, vn, kc, vc, c.seqlens, c.block_table, s.B, c.s_new, s.Hk,
                                                           c.cap, c.num_pages, c.page_size, c.max_pages, c.rot);
      break;
    case 256:
      fa_kv_append_kernel<256><<<grid, 256, 0, stream>>>(kn, vn, kc, vc, c.seqlens, c.block_table, s.B, c.s_new, s.Hk,
                                                           c.cap, c.num_pages, c.page_size, c.max_pages, c.rot);
      break;
    default:
      return FA_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t decode_workspace_bytes(int B, int Sq, int H, int D, int n) {
  const size_t units = size_t(B) * Sq * H * n;
  return align256(units * D * 4) + align256(units * 4);
}

// Query pairs a split CTA serves: up to four, as many as one key/value head has.
static int decode_rows_per_cta(int Sq, int H, int Hk) {
  const int pairs = Sq * (H / Hk);
  return pairs >= 4 ? 4 : (pairs >= 2 ? 2 : 1);
}

int decode_auto_splits(int B, int Sq, int Sk, int H, int Hk, int D) {
  const int tk = (D == 64) ? 128 : (D == 128 ? 64 : 32);
  const long long slots = 2LL * device_sm_count();  // two split CTAs fit per SM
  const int rpc = decode_rows_per_cta(Sq, H, Hk);
  const long long units = (long long)B * Hk * ((Sq * (H / Hk) + rpc - 1) / rpc);  // CTAs per split
  int max_n = (Sk + 4 * tk - 1) / (4 * tk);  // at least four tiles per split
  if (max_n < 1) max_n = 1;
  if (max_n > 256) max_n = 256;
  int best = 1;
  double best_eff = 0.0;
  for (int n = 1; n <= max_n; ++n) {
    const long long ctas = units * n;
    const long long waves = (ctas + slots - 1) / slots;
    const double eff = double(ctas) / double(waves * slots);
    if (eff >= 0.95) return n;
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = n;
    }
  }
  return best;
}

template <int D>
static int launch_decode_t(const AttnShape& s, const void* q, const void* k, const void* v, void* out, float* lse,
                           void* ws, int n, const CacheArgs* cg, cudaStream_t stream) {
  using C = DecCfg<D>;
  const bool paged = cg && cg->block_table;
  if (paged && cg->page_size % C::TK != 0) return FA_ERR_UNSUPPORTED;
  // Dense caches are (B, rows, Hk, D); pages are (num_pages, page_size, Hk, D).
  const int mb = paged ? cg->num_pages : s.B, mrows = paged ? cg->page_size : (cg ? cg->cap : s.Sk);
  CUtensorMap mk, mv;
  if (!make_bshd_map(&mk, k, mb, mrows, s.Hk, D, C::TK) || !make_bshd_map(&mv, v, mb, mrows, s.Hk, D, C::TK))
    return FA_ERR_CUDA;
  const int rpc = decode_rows_per_cta(s.Sq, s.H, s.Hk);
  auto kern = rpc == 4 ? fa_decode_split_kernel<D, 4> : (rpc == 2 ? fa_decode_split_kernel<D, 2> : fa_decode_split_kernel<D, 1>);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
    return FA_ERR_CUDA;
  DecParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  const size_t units = size_t(s.B) * s.Sq * s.H * n;
  p.part_o = static_cast<float*>(ws);
  p.part_l = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + align256(units * D * 4));
  p.alibi = s.alibi;
  p.alibi_bstride = s.alibi_bstride;
  p.B = s.B;
  p.Sq = s.Sq;
  p.Sk = s.Sk;
  p.H = s.H;
  p.group = s.H / s.Hk;
  p.n_rb = (s.Sq * p.group + rpc - 1) / rpc;
  p.block_table = cg ? cg->block_table : nullptr;
  p.seqlens_k = cg ? cg->seqlens : nullptr;
  p.page_size = cg ? cg->page_size : 0;
  p.max_pages = cg ? cg->max_pages : 0;
  p.s_new = cg ? cg->s_new : 0;
  p.cap = cg ? cg->cap : s.Sk;
  p.rot = cg ? cg->rot : Rotary{nullptr, nullptr, 0, 0, 0};
  p.n_splits = n;
  p.wl = s.wl;
  p.wr = s.wr;
  p.scale_log2 = s.scale * 1.4426950408889634f;
  p.status = device_status_word();
  if (!p.status) return FA_ERR_CUDA;
  if (s.B > 65535 || (long long)s.Hk * p.n_rb > 65535) return FA_ERR_UNSUPPORTED;
  dim3 grid(n, s.Hk * p.n_rb, s.B);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(mk, mv, p);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  const int warps = s.B * s.Sq * s.H;
  fa_decode_combine_kernel<D><<<(warps + 7) / 8, 256, 0, stream>>>(
      p.part_o, p.part_l, static_cast<__nv_bfloat16*>(out), lse, s.B, s.Sq, s.H, n);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int decode_launch(const AttnShape& s, const void* q, const void* k, const void* v, void* out, float* lse,
                  void* workspace, int n, const CacheArgs* paged, cudaStream_t stream) {
  switch (s.D) {
    case 64:
      return launch_decode_t<64>(s, q, k, v, out, lse, workspace, n, paged, stream);
    case 128:
      return launch_decode_t<128>(s, q, k, v, out, lse, workspace, n, paged, stream);
    case 256:
      return launch_decode_t<256>(s, q, k, v, out, lse, workspace, n, paged, stream);
    default:
      return FA_ERR_UNSUPPORTED;
  }
}

}  // namespace fa
