// Split-KV decode for short queries: two split kernels (CUDA cores for up to
// three query pairs per key/value head, tensor cores from four on), the query
// rotation the tensor-core kernel reads, the KV-cache append, and the merge
// kernel.
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
// Tensor-core split kernel (fa_decode_mma_kernel, described where it is
// defined): the pairs of one key/value head as the rows of a 128-row MMA tile.
// Merge kernel (one block of four warps per (batch, query row, head)):
//   L = log sum_s exp(L_s), O = sum_s exp(L_s - L) O_s.
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
  int n_rb;   // CTAs (row blocks) per key/value head and split
  int rows_i; // tensor-core kernel: query rows per block (rows_i * group <= 128)
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
  uint64_t wait_ns;  // bounded-wait limit
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
  const Watch watch{&bars->abort, p.status, p.wait_ns};

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
            if (globaltimer_ns() - t0 > p.wait_ns) break;
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


// ============================================================================ grouped decode on tensor cores
// The (query row, query head) pairs that read one key/value head are the rows
// of one 128-row MMA tile (row r: query row i0 + r / group, query head
// hk * group + r % group, one TMA box of group heads x rows_i rows). Per key
// tile, as in the forward kernel: S = Q K^T into TMEM (two buffers), an online
// softmax with one thread per row (its own mask, ALiBi slope and diagonal),
// P (bf16) written over S, O += P V. Each K/V tile is read once for all the
// pairs; the split's normalised O_s and L_s go to the same partials the merge
// kernel reads.
// ROT: the query was rotated (rotary) in fp32 by a separate kernel and comes as a
// bf16 pair q_hi + q_lo (q_lo = the rounding residual), two Q tiles whose
// products with K accumulate in fp32: S keeps about 16 bits of the rotated q
// rather than bf16's 8.
template <int D, bool ROT = false>
struct DecMmaCfg {
  static constexpr int PANELS = D / 64;
  static constexpr int PANEL_BYTES = 128 * 128;
  static constexpr int TILE_BYTES = PANELS * PANEL_BYTES;  // 128 rows (or keys) x D
  static constexpr int TK = 128;                           // keys per tile
  // Softmax warpgroups: two where TMEM holds two O accumulators (D <= 128);
  // group w takes the CTA's key tiles w, w + NW, ... with its own S buffer and O,
  // and the two running states are merged exactly at the end.
  static constexpr int NW = D <= 128 ? 2 : 1;
  static constexpr int NQ = ROT ? 2 : 1;                   // Q tiles (q_hi, q_lo)
  static constexpr int NSLOT = D == 64 ? 8 : (D == 128 ? (ROT ? 5 : 6) : 2);  // ring of K_j, V_j tiles
  static constexpr int THREADS = 128 + 128 * NW;           // producer, MMA, 2 idle, softmax warps
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = NQ * TILE_BYTES;
  static constexpr int BAR_OFF = KV_OFF + NSLOT * TILE_BYTES;
  static constexpr int XCH_OFF = BAR_OFF + 256;            // group 1's (m, l) per row for the merge
  static constexpr int SMEM_BYTES = XCH_OFF + 1024 + 1024;  // + alignment slack
  static constexpr uint32_t O_COL0 = 256;                  // TMEM: S buffers at 0 and 128, O after
  static_assert(O_COL0 + NW * D <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct DecMmaBars {
  uint64_t q_full;
  uint64_t kv_full[8], kv_empty[8];
  uint64_t s_full[2], p_full[2];  // per S buffer (P is written over its S)
  uint64_t pv_done[2], o_done[2];  // per softmax group
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(DecMmaBars) <= 256, "barrier block");

enum : uint32_t {
  SITE_DM_EMPTY = 0x61,
  SITE_DM_Q = 0x62,
  SITE_DM_K = 0x63,
  SITE_DM_V = 0x64,
  SITE_DM_P = 0x65,
  SITE_DM_S = 0x66,
  SITE_DM_PV = 0x67,
  SITE_DM_EPI = 0x68,
};

// Timeout-only wait used while draining after an abort.
__device__ __forceinline__ void dm_drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

template <int D, bool ROT>
__global__ void __launch_bounds__(DecMmaCfg<D, ROT>::THREADS, 1)
    fa_decode_mma_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_q_lo,
                         const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const DecParams p) {
  using C = DecMmaCfg<D, ROT>;
  constexpr int NW = C::NW;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  DecMmaBars* bars = reinterpret_cast<DecMmaBars*>(smem + C::BAR_OFF);
  float* xch_m = reinterpret_cast<float*>(smem + C::XCH_OFF);  // [128]
  float* xch_l = xch_m + 128;                                  // [128]
  const int warp = int(warp_id());
  const int lane = int(lane_id());

  const int split = blockIdx.x;
  const int hk = blockIdx.y / p.n_rb;
  const int rb = blockIdx.y % p.n_rb;
  const int b = blockIdx.z;
  const int i0 = rb * p.rows_i;                   // first query row of this block
  const int i1 = min(p.Sq, i0 + p.rows_i) - 1;    // last
  // this sequence's keys, clamped to what the cache (or its page table) holds
  const int Sk = p.seqlens_k ? max(0, min(p.seqlens_k[b] + p.s_new, p.cap)) : p.Sk;
  // The split's whole tiles; the rows' live bounds grow with the row, so the
  // first and last rows bound the keys any row of the block can see.
  const int n_all = (Sk + C::TK - 1) / C::TK;
  const int s_lo = int((long long)n_all * split / p.n_splits) * C::TK;
  const int s_hi = min(Sk, int((long long)n_all * (split + 1) / p.n_splits) * C::TK);  // exclusive
  const int ks = max(s_lo, live_range(i0, p.Sq, Sk, p.wl, p.wr).lo);
  const int ke = min(s_hi, live_range(i1, p.Sq, Sk, p.wl, p.wr).hi + 1);
  const int t0 = (ks / C::TK) * C::TK;
  const int n_blocks = ke > ks ? (ke - t0 + C::TK - 1) / C::TK : 0;
  // key tiles of softmax group w: w, w + NW, ...
  auto tiles_of = [&](int w) { return n_blocks > w ? (n_blocks - w + NW - 1) / NW : 0; };
  // First key of tile jj. A decode row's diagonal key lies at the end of the
  // cache, where ALiBi's bias peaks, so with ALiBi the tiles run from the last
  // one down: the running max is set by the first tile and O is rarely rescaled.
  const bool rev = p.alibi != nullptr;
  auto key_row = [t0, n_blocks, rev](int jj) { return t0 + (rev ? n_blocks - 1 - jj : jj) * C::TK; };

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->p_full[s], 4);  // one arrive per softmax warp
      mbar_init(&bars->pv_done[s], 1);
      mbar_init(&bars->o_done[s], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const Watch watch{&bars->abort, p.status, p.wait_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop; one elected lane issues each copy.
    if (n_blocks > 0) {
      tma_prefetch_desc_w(&tm_q);
      if (ROT) tma_prefetch_desc_w(&tm_q_lo);
      tma_prefetch_desc_w(&tm_k);
      tma_prefetch_desc_w(&tm_v);
      // one box per 64-column panel: group heads x rows_i query rows (rows past
      // Sq read zeros); the tile's rows past group * rows_i are never read back
      mbar_arrive_expect_tx_w(&bars->q_full, C::NQ * C::PANELS * 128 * p.group * p.rows_i);
      for (int pn = 0; pn < C::PANELS; ++pn) {
        tma_load_4d_w(smem + C::Q_OFF + pn * C::PANEL_BYTES, &tm_q, &bars->q_full, pn * 64, hk * p.group, i0, b);
        if (ROT)
          tma_load_4d_w(smem + C::Q_OFF + C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_q_lo, &bars->q_full, pn * 64,
                        hk * p.group, i0, b);
      }
      int issued = 0;
      bool ok = true;
      for (int jj = 0; jj < n_blocks && ok; ++jj) {
        int row = key_row(jj), tb = b;
        if (p.block_table) {  // (row in page, page) coordinates of this tile
          tb = p.block_table[size_t(b) * p.max_pages + row / p.page_size];
          row %= p.page_size;
        }
        for (int kv = 0; kv < 2; ++kv) {
          const int it = 2 * jj + kv;
          const int s = it % C::NSLOT;
          if (!fa_wait_warp(&bars->kv_empty[s], (uint32_t(it / C::NSLOT) & 1u) ^ 1u, watch, SITE_DM_EMPTY)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx_w(&bars->kv_full[s], C::TILE_BYTES);
          const CUtensorMap* m = kv ? &tm_v : &tm_k;
          for (int pn = 0; pn < C::PANELS; ++pn)
            tma_load_4d_w(smem + C::KV_OFF + s * C::TILE_BYTES + pn * C::PANEL_BYTES, m, &bars->kv_full[s],
                          pn * 64, hk, row, tb);
          issued = it + 1;
        }
      }
      if (!ok) {  // let the copies in flight land before the CTA leaves
        dm_drain_wait(&bars->q_full, 0, p.wait_ns);
        for (int it = (issued > C::NSLOT ? issued - C::NSLOT : 0); it < issued; ++it)
          dm_drain_wait(&bars->kv_full[it % C::NSLOT], uint32_t(it / C::NSLOT) & 1u, p.wait_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop; one elected lane issues each MMA and commit.
    if (n_blocks > 0) {
      constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, 0, 0);  // Q, K both K-major
      constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, 0, 1);    // P from TMEM, V MN-major
      const uint64_t q_desc = sdesc_sw128(smem_u32(smem + C::Q_OFF), 16, 1024);
      const uint64_t kv_kdesc = sdesc_sw128(smem_u32(smem + C::KV_OFF), 16, 1024);
      const uint64_t kv_mdesc = sdesc_sw128(smem_u32(smem + C::KV_OFF), C::PANEL_BYTES, 1024);
      auto slot_of = [](int it) { return it % C::NSLOT; };
      auto wait_full = [&](int it, uint32_t site) {
        return fa_wait_warp(&bars->kv_full[slot_of(it)], uint32_t(it / C::NSLOT) & 1u, watch, site);
      };
      auto issue_s = [&](int jj, int sb) {  // S of key tile jj into S buffer sb
        if (!wait_full(2 * jj, SITE_DM_K)) return false;
        tc_fence_after();
        const uint64_t kd = sdesc_adv(kv_kdesc, uint32_t(slot_of(2 * jj)) * C::TILE_BYTES);
        const uint32_t ts = tmem + uint32_t(sb) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::PANEL_BYTES + (kk % 4) * 32;
          mma_ss_w(ts, sdesc_adv(q_desc, off), sdesc_adv(kd, off), IDESC_S, kk > 0 ? 1u : 0u);
        }
        if (ROT) {  // + q_lo K^T, accumulated
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = C::TILE_BYTES + (kk / 4) * C::PANEL_BYTES + (kk % 4) * 32;
            mma_ss_w(ts, sdesc_adv(q_desc, off), sdesc_adv(kd, off - C::TILE_BYTES), IDESC_S, 1u);
          }
        }
        mma_commit_w(&bars->s_full[sb]);
        mma_commit_w(&bars->kv_empty[slot_of(2 * jj)]);
        return true;
      };
      // PV of key tile jj for softmax group w = jj % NW, P read from S buffer sb
      auto issue_pv = [&](int jj, int sb, uint32_t p_parity) {
        const int w = jj % NW, j = jj / NW;  // group and its local tile index
        if (!wait_full(2 * jj + 1, SITE_DM_V)) return false;
        if (!fa_wait_warp(&bars->p_full[sb], p_parity, watch, SITE_DM_P)) return false;
        tc_fence_after();
        const uint64_t vd = sdesc_adv(kv_mdesc, uint32_t(slot_of(2 * jj + 1)) * C::TILE_BYTES);
        const uint32_t to = tmem + C::O_COL0 + uint32_t(w) * D, tp = tmem + uint32_t(sb) * 128;
        const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ts_w(to, tp + kk * 8, sdesc_adv(vd, kk * 2048), IDESC_O, kk > 0 ? 1u : acc0);
        mma_commit_w(&bars->pv_done[w]);
        if (j == tiles_of(w) - 1) mma_commit_w(&bars->o_done[w]);  // the group's last PV
        mma_commit_w(&bars->kv_empty[slot_of(2 * jj + 1)]);
        return true;
      };
      bool ok = fa_wait_warp(&bars->q_full, 0, watch, SITE_DM_Q);
      if (NW == 2) {
        // Per pair of tiles: S_0(a), PV_1(a - 1), S_1(a + 1), PV_0(a) (a = 2j): each
        // group's S overwrites its own P, read by its PV issued before (in order),
        // and each group has the other's MMAs' worth of time per tile.
        for (int a = 0; a < n_blocks && ok; a += 2) {
          if (!(ok = issue_s(a, 0))) break;
          if (a > 0 && !(ok = issue_pv(a - 1, 1, uint32_t((a - 1) / 2) & 1u))) break;
          if (a + 1 < n_blocks && !(ok = issue_s(a + 1, 1))) break;
          if (!(ok = issue_pv(a, 0, uint32_t(a / 2) & 1u))) break;
        }
        // the loop issued PV_1 of every odd tile but the last one when the count is even
        if (ok && n_blocks % 2 == 0) ok = issue_pv(n_blocks - 1, 1, uint32_t((n_blocks - 1) / 2) & 1u);
      } else {
        // One group, two S buffers: S(jj+1) into the other buffer as soon as K(jj+1)
        // is in; it overwrites P(jj-1), read by PV(jj-1) before (in order). P
        // barriers are per buffer: S(jj+1) is queued before PV(jj)'s wait, so the
        // softmax may finish tile jj+1 first; buffer jj & 1 is next used by S(jj+2).
        ok = ok && issue_s(0, 0);
        for (int jj = 0; jj < n_blocks && ok; ++jj) {
          if (jj + 1 < n_blocks && !(ok = issue_s(jj + 1, (jj + 1) & 1))) break;
          if (!(ok = issue_pv(jj, jj & 1, uint32_t(jj >> 1) & 1u))) break;
        }
      }
      if (!ok) {  // let issued MMAs finish before TMEM is released
        mma_commit_w(&bars->drain);
        dm_drain_wait(&bars->drain, 0, p.wait_ns);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax (thread = pair)
    const int w = (warp - 4) / 4;  // softmax group
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_addr = uint32_t(wq * 32) << 16;
    const int i = i0 + r / p.group;               // query row of this pair
    const int h = hk * p.group + r % p.group;     // query head of this pair
    const bool pair_ok = r < p.rows_i * p.group && i < p.Sq;
    // this pair's keys: its live range clipped to the split
    int klo = 1, khi = 0;
    if (pair_ok) {
      const RowRange rr = live_range(i, p.Sq, Sk, p.wl, p.wr);
      klo = max(s_lo, rr.lo);
      khi = min(s_hi, rr.hi + 1);
    }
    const bool has_alibi = p.alibi != nullptr;
    const float slope_log2 = (has_alibi && pair_ok) ? p.alibi[b * p.alibi_bstride + h] * 1.4426950408889634f : 0.0f;
    const int c_i = i + Sk - p.Sq;
    const float sl = p.scale_log2;
    const uint32_t o_col = C::O_COL0 + uint32_t(w) * D;

    float m = -INFINITY;  // reference max (log2 units) the running O and l are relative to
    float l = 0.0f;
    bool ok = true;
    const int n_mine = tiles_of(w);
    for (int j = 0; j < n_mine; ++j) {
      const int jj = j * NW + w;  // key tile
      const int sb = (NW == 2) ? w : (j & 1);
      const uint32_t par = (NW == 2) ? (uint32_t(j) & 1u) : (uint32_t(j >> 1) & 1u);
      if (!(ok = fa_wait_warp(&bars->s_full[sb], par, watch, SITE_DM_S))) break;
      tc_fence_after();
      float x[128];
      tmem_ld_x128f(tmem + lane_addr + uint32_t(sb) * 128, x);
      const int kbase = key_row(jj);
      if (has_alibi) {
        // x = scale*log2(e)*qk - slope*log2(e)*|c(i) - j|, in log2 units
        const float d0 = float(c_i - kbase);
        if (kbase + 127 <= c_i || kbase >= c_i) {
          // keys on one side of the diagonal: the bias on column pairs with the
          // signed slope (the distances are exact integers)
          const float ns = (kbase >= c_i) ? slope_log2 : -slope_log2;
          const uint64_t ns2 = f2_pack(ns, ns), sl2 = f2_pack(sl, sl), st2 = f2_pack(8.0f, 8.0f);
          uint64_t dist[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) dist[k] = f2_pack(d0 - float(2 * k), d0 - float(2 * k + 1));
#pragma unroll
          for (int c = 0; c < 128; c += 8) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int cc = c + 2 * k;
              f2_unpack(f2_fma(f2_pack(x[cc], x[cc + 1]), sl2, f2_mul(dist[k], ns2)), x[cc], x[cc + 1]);
              dist[k] = f2_sub(dist[k], st2);
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 128; ++c) x[c] = fmaf(x[c], sl, -slope_log2 * fabsf(d0 - float(c)));
        }
      }
      // keys outside this pair's [klo, khi) are masked; a tile inside it needs no mask
      if (!(kbase >= klo && kbase + 127 < khi)) {
        const int lo = klo - kbase, hi = khi - kbase;
#pragma unroll
        for (int c = 0; c < 128; ++c) x[c] = (c >= lo && c < hi) ? x[c] : -INFINITY;
      }
      float mq[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) mq[k] = fmaxf(x[2 * k], x[2 * k + 1]);
#pragma unroll
      for (int c = 8; c < 128; c += 8) {
#pragma unroll
        for (int k = 0; k < 4; ++k) mq[k] = max3f(mq[k], x[c + 2 * k], x[c + 2 * k + 1]);
      }
      const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      // block max in log2 units (without ALiBi, x still holds raw q.k and scale > 0)
      const float m_blk = has_alibi ? mx : mx * sl;
      const float m_new = fmaxf(m, m_blk);
      float alpha = 1.0f;
      if (m_new != -INFINITY) {
        if (m == -INFINITY) {
          m = m_new;  // first live key: O and l are still exactly 0
        } else if (m_new > m + 8.0f) {
          alpha = ex2_approx(m - m_new);
          m = m_new;
        }
      }
      l *= alpha;
      const float m_use = (m == -INFINITY) ? 0.0f : m;
      // p = 2^(x*sl - m) without ALiBi; with ALiBi x is already in log2 units.
      // Column pairs go through the paired FMA and add; rs2[k] sums the pairs
      // e with e % 2 == k.
      const float mul = has_alibi ? 1.0f : sl;
      const uint64_t mul2 = f2_pack(mul, mul), nm2 = f2_pack(-m_use, -m_use);
      uint64_t rs2[2] = {f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f)};
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c = q4 * 32 + 2 * e;
          float a0, a1;
          f2_unpack(f2_fma(f2_pack(x[c], x[c + 1]), mul2, nm2), a0, a1);
          const float p0 = ex2_approx(a0);
          const float p1 = ex2_approx(a1);
          rs2[e & 1] = f2_add(rs2[e & 1], f2_pack(p0, p1));
          pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st_x16(tmem + lane_addr + uint32_t(sb) * 128 + q4 * 16, pk);
      }
      {
        float r0, r1, r2, r3;
        f2_unpack(rs2[0], r0, r1);
        f2_unpack(rs2[1], r2, r3);
        l += (r0 + r1) + (r2 + r3);
      }
      if (__any_sync(0xffffffffu, alpha != 1.0f) && j > 0) {
        // O must hold this group's P V of its previous tile before it is rescaled.
        if (!(ok = fa_wait_warp(&bars->pv_done[w], uint32_t(j - 1) & 1u, watch, SITE_DM_PV))) break;
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          const uint32_t oa = tmem + lane_addr + o_col + cc * 32;
          tmem_ld_x32(oa, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st_x32(oa, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(&bars->p_full[sb]);
    }

    // ------------------------------------------------------------ partials of this split
    // Group 1 hands its (m, l) to group 0, which merges the two states exactly
    // (O rows of both groups sit in the same TMEM lanes) and writes O_s, L_s.
    if (NW == 2) {
      if (w == 1) {
        xch_m[r] = ok ? m : -INFINITY;
        xch_l[r] = ok ? l : 0.0f;
      }
      named_bar_sync(2, 256);
    }
    if (w == 0) {
      const size_t pidx = ((size_t(b) * p.Sq + (pair_ok ? i : 0)) * p.H + h) * p.n_splits + split;
      const float m1 = (NW == 2) ? xch_m[r] : -INFINITY;
      const float l1 = (NW == 2) ? xch_l[r] : 0.0f;
      bool done = ok && (n_mine == 0 || fa_wait_warp(&bars->o_done[0], 0, watch, SITE_DM_EPI));
      if (NW == 2 && tiles_of(1) > 0) done = done && fa_wait_warp(&bars->o_done[1], 0, watch, SITE_DM_EPI);
      if (done) {
        tc_fence_after();
        const float M = fmaxf(m, m1);
        const float w0 = (m == -INFINITY) ? 0.0f : ex2_approx(m - M);
        const float w1 = (m1 == -INFINITY) ? 0.0f : ex2_approx(m1 - M);
        const float L = l * w0 + l1 * w1;
        const float inv = (L > 0.0f) ? 1.0f / L : 0.0f;
        const bool use0 = m != -INFINITY, use1 = m1 != -INFINITY;  // a group with no live key has no O
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o0[32], o1[32];
          tmem_ld_x32(tmem + lane_addr + C::O_COL0 + cc * 32, o0);
          if (NW == 2) tmem_ld_x32(tmem + lane_addr + C::O_COL0 + D + cc * 32, o1);
          if (pair_ok) {
            float v[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              float acc = use0 ? __uint_as_float(o0[e]) * w0 : 0.0f;
              if (NW == 2 && use1) acc += __uint_as_float(o1[e]) * w1;
              v[e] = acc * inv;
            }
            float4* dst = reinterpret_cast<float4*>(p.part_o + pidx * D + cc * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e) dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
          }
        }
        if (pair_ok) p.part_l[pidx] = (L > 0.0f) ? (M + lg2_approx(L)) * 0.6931471805599453f : -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
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

// Merge of the splits' partials (section "2.2" of the page cited at the top of
// this file): out = sum_s e^(L_s - L) O_s with L = log sum_s e^(L_s). One block of four warps per (b, query row, head); the
// 128 threads read the L_s (n <= 256, two per thread), warp w folds the splits
// s = w, w + 4, ... with independent loads in flight, and the four sums meet in
// shared memory. A split with no live key wrote O_s = 0 and L_s = -inf.
constexpr int COMBINE_THREADS = 128;
template <int D>
__global__ void __launch_bounds__(COMBINE_THREADS) fa_decode_combine_kernel(const float* __restrict__ part_o,
                                                                             const float* __restrict__ part_l,
                                                                             __nv_bfloat16* __restrict__ out,
                                                                             float* __restrict__ lse, int Sq, int H,
                                                                             int n) {
  constexpr int PER = D / 32;  // columns per lane: 2, 4 or 8
  constexpr int NWARP = COMBINE_THREADS / 32;
  __shared__ float red[NWARP];
  __shared__ float acc_s[NWARP - 1][D];
  const int row = blockIdx.x;  // (b * Sq + i) * H + h
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t base = size_t(row) * n;
  const float l0 = tid < n ? part_l[base + tid] : -INFINITY;
  const float l1 = tid + COMBINE_THREADS < n ? part_l[base + tid + COMBINE_THREADS] : -INFINITY;
  float M = fmaxf(l0, l1);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int w = 1; w < NWARP; ++w) M = fmaxf(M, red[w]);
  const float Ms = (M == -INFINITY) ? 0.0f : M;
  float Z = ((l0 == -INFINITY) ? 0.0f : __expf(l0 - Ms)) + ((l1 == -INFINITY) ? 0.0f : __expf(l1 - Ms));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, off);
  __syncthreads();  // every thread has read red[] as maxima
  if (lane == 0) red[warp] = Z;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.0f;
#pragma unroll 4
  for (int s = warp; s < n; s += NWARP) {
    const float ls = part_l[base + s];
    const float* src = part_o + (base + s) * D + lane * PER;
    float v[PER];
#pragma unroll
    for (int e = 0; e < PER; e += 2) {
      const float2 v2 = *reinterpret_cast<const float2*>(src + e);
      v[e] = v2.x;
      v[e + 1] = v2.y;
    }
    const float w = (ls == -INFINITY) ? 0.0f : __expf(ls - Ms);
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, v[e], acc[e]);
  }
  if (warp > 0) {
#pragma unroll
    for (int e = 0; e < PER; ++e) acc_s[warp - 1][lane * PER + e] = acc[e];
  }
  __syncthreads();
  if (warp != 0) return;
  Z = red[0];
#pragma unroll
  for (int w = 1; w < NWARP; ++w) Z += red[w];
  const float invZ = Z > 0.0f ? 1.0f / Z : 0.0f;
#pragma unroll
  for (int w = 0; w < NWARP - 1; ++w) {
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] += acc_s[w][lane * PER + e];
  }
  uint32_t pk[PER / 2];
#pragma unroll
  for (int e = 0; e < PER / 2; ++e) pk[e] = pack_bf16x2(acc[2 * e] * invZ, acc[2 * e + 1] * invZ);
  __nv_bfloat16* dst = out + size_t(row) * D + lane * PER;  // out is (B, Sq, H, D)
  if constexpr (PER == 2) {
    *reinterpret_cast<uint32_t*>(dst) = pk[0];
  } else if constexpr (PER == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(pk[0], pk[1]);
  } else {
    *reinterpret_cast<uint4*>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
  if (lane == 0) {
    const int h = row % H, i = (row / H) % Sq, b = row / (H * Sq);
    lse[(size_t(b) * H + h) * Sq + i] = (Z > 0.0f) ? Ms + __logf(Z) : -INFINITY;
  }
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

// Workspace: the split partials O_s (fp32) and L_s, then room for the rotated
// query as a bf16 pair q_hi, q_lo (the tensor-core kernel's query tile arrives
// by TMA, so rotary is applied before it, into these copies).
size_t decode_workspace_bytes(int B, int Sq, int H, int D, int n, bool with_rotary) {
  const size_t units = size_t(B) * Sq * H * n;
  const size_t part = align256(units * D * 4) + align256(units * 4);
  return with_rotary ? part + 2 * align256(size_t(B) * Sq * H * D * 2) : part;
}

// Rotary of the queries for the tensor-core decode: q rotated in fp32 at each
// row's diagonal position i + Sk_b - Sq (as the CUDA-core kernel does in
// registers), stored as q_hi = bf16(q_rot) and q_lo = bf16(q_rot - q_hi); one
// thread per 16-byte chunk.
template <int D>
__global__ void __launch_bounds__(256)
    fa_decode_rotate_q_kernel(const __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ q_hi,
                              __nv_bfloat16* __restrict__ q_lo, const int* __restrict__ seqlens, int B, int Sq,
                              int H, int Sk, int s_new, int cap, Rotary rot) {
  constexpr int CH = D / 8;
  const long long n = (long long)B * Sq * H * CH;
  for (long long t = blockIdx.x * 256LL + threadIdx.x; t < n; t += (long long)gridDim.x * 256) {
    const int c = int(t % CH);
    const long long row = t / CH;  // (b, i, h)
    const int i = int((row / H) % Sq);
    const int b = int(row / ((long long)H * Sq));
    const int skb = seqlens ? max(0, min(seqlens[b] + s_new, cap)) : Sk;
    const __nv_bfloat16* src = q + row * D;
    float x[8], pq[8];
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(src + c * 8), x);
    if (c * 8 < rot.dim) {
      if (!rot.interleaved) bf16x8_to_f32(*reinterpret_cast<const uint4*>(src + rotary_partner(c * 8, rot)), pq);
      rotary8(x, pq, c * 8, i + skb - Sq, rot);
    }
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      hi[e] = pack_bf16x2(x[2 * e], x[2 * e + 1]);
      const float h0 = __uint_as_float(hi[e] << 16), h1 = __uint_as_float(hi[e] & 0xFFFF0000u);
      lo[e] = pack_bf16x2(x[2 * e] - h0, x[2 * e + 1] - h1);
    }
    *reinterpret_cast<uint4*>(q_hi + row * D + c * 8) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(q_lo + row * D + c * 8) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// Query pairs a split CTA serves: up to four, as many as one key/value head has.
static int decode_rows_per_cta(int Sq, int H, int Hk) {
  const int pairs = Sq * (H / Hk);
  return pairs >= 4 ? 4 : (pairs >= 2 ? 2 : 1);
}

// The tensor-core kernel serves a key/value head's pairs as the rows of one
// MMA tile: worth it from 4 pairs on (fewer pairs leave the CUDA-core kernel
// bound by the cache read), possible while one query row's group heads fit the
// 128 rows.
static bool decode_mma_ok(int Sq, int H, int Hk) {
  const int g = H / Hk;
  return g <= 128 && Sq * g >= 4;
}
static int decode_mma_rows(int Sq, int H, int Hk) {  // query rows per block
  return std::min(Sq, 128 / (H / Hk));
}
// The split kernel the launcher runs: the tensor-core one unless the pages
// are smaller than its 128-key tiles or rotary is asked for at D = 256 (its
// two query tiles leave no room for the K/V ring).
static bool decode_uses_mma(const AttnShape& s, const CacheArgs* cg) {
  const bool paged = cg && cg->block_table;
  const bool rot = cg && cg->rot.cos;
  return decode_mma_ok(s.Sq, s.H, s.Hk) && !(paged && cg->page_size % DecMmaCfg<64>::TK != 0) &&
         !(rot && s.D > 128);
}

int decode_check(const AttnShape& s, const CacheArgs* cg) {
  long long blocks;  // gridDim.y = Hk x blocks of query pairs
  if (decode_uses_mma(s, cg)) {
    const int rows_i = decode_mma_rows(s.Sq, s.H, s.Hk);
    blocks = (s.Sq + rows_i - 1) / rows_i;
  } else {
    const int rpc = decode_rows_per_cta(s.Sq, s.H, s.Hk);
    blocks = ((long long)s.Sq * (s.H / s.Hk) + rpc - 1) / rpc;
  }
  if (s.B > 65535 || (long long)s.Hk * blocks > 65535) return FA_ERR_UNSUPPORTED;
  // the combine kernel numbers the (batch, query row, head) triples with 32-bit ints
  if ((long long)s.B * s.Sq * s.H > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

int decode_auto_splits(int B, int Sq, int Sk, int H, int Hk, int D) {
  const bool mma = decode_mma_ok(Sq, H, Hk);
  const int tk = mma ? 128 : ((D == 64) ? 128 : (D == 128 ? 64 : 32));
  const long long sms = device_sm_count();
  const long long slots = (mma ? 1LL : 2LL) * sms;  // CTAs that fit per SM
  const int rpc = decode_rows_per_cta(Sq, H, Hk);
  const int rows_i = decode_mma_rows(Sq, H, Hk);
  const long long units = mma ? (long long)B * Hk * ((Sq + rows_i - 1) / rows_i)  // CTAs per split
                              : (long long)B * Hk * ((Sq * (H / Hk) + rpc - 1) / rpc);
  // at least four tiles per split
  int max_n = (Sk + 4 * tk - 1) / (4 * tk);
  if (max_n < 1) max_n = 1;
  if (max_n > 256) max_n = 256;
  if (mma) {
    // Tensor-core kernel (one CTA per SM): about 0.85 x the SM count of its CTAs
    // already draw the whole HBM bandwidth on a long cache (measured on 152
    // SMs: 128 CTAs beat 144 and 152, and every split count making more CTAs
    // than that in one wave, or a second wave, only adds a tail). With fewer
    // units than that, the largest split count staying within it.
    const long long fill = std::max(1LL, sms * 85 / 100);
    if (units <= fill) return int(std::max(1LL, std::min<long long>(max_n, fill / units)));
  }
  // Otherwise the fewest splits that fill whole waves to 95%, else the best fill.
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
  // Tensor-core path: pairs of a key/value head as MMA rows (decode_uses_mma).
  static_assert(DecMmaCfg<D>::TK == DecMmaCfg<64>::TK, "one key tile for every D");
  const bool rot = cg && cg->rot.cos;
  const bool mma = decode_uses_mma(s, cg);
  {
    const int st = decode_check(s, cg);
    if (st != FA_OK) return st;
  }
  if (paged && cg->page_size % C::TK != 0) return FA_ERR_UNSUPPORTED;
  // Dense caches are (B, rows, Hk, D); pages are (num_pages, page_size, Hk, D).
  const int mb = paged ? cg->num_pages : s.B, mrows = paged ? cg->page_size : (cg ? cg->cap : s.Sk);
  CUtensorMap mk, mv;
  if (!make_bshd_map(&mk, k, mb, mrows, s.Hk, D, C::TK) || !make_bshd_map(&mv, v, mb, mrows, s.Hk, D, C::TK))
    return FA_ERR_CUDA;
  const int rpc = decode_rows_per_cta(s.Sq, s.H, s.Hk);
  auto kern = rpc == 4 ? fa_decode_split_kernel<D, 4> : (rpc == 2 ? fa_decode_split_kernel<D, 2> : fa_decode_split_kernel<D, 1>);
  if (!mma && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
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
  p.rows_i = 0;  // tensor-core kernel only
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
  p.wait_ns = debug_settings().wait_ns;
  if (!p.status) return FA_ERR_CUDA;
  if (mma) {
    using M = DecMmaCfg<D>;
    p.rows_i = decode_mma_rows(s.Sq, s.H, s.Hk);
    p.n_rb = (s.Sq + p.rows_i - 1) / p.rows_i;
    // with rotary, the query tiles come from the rotated pair in the workspace
    const void* qsrc = q;
    const void* qlo = q;
    if (rot) {
      const size_t qbytes = align256(size_t(s.B) * s.Sq * s.H * D * 2);
      auto* qh = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(ws) + align256(units * D * 4) +
                                                  align256(units * 4));
      auto* ql = reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<uint8_t*>(qh) + qbytes);
      const long long chunks = (long long)s.B * s.Sq * s.H * (D / 8);
      const int rgrid = int(std::max(1LL, std::min((long long)device_sm_count() * 8, (chunks + 255) / 256)));
      fa_decode_rotate_q_kernel<D><<<rgrid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(q), qh, ql,
                                                               p.seqlens_k, s.B, s.Sq, s.H, s.Sk, p.s_new, p.cap,
                                                               p.rot);
      if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
      qsrc = qh;
      qlo = ql;
    }
    CUtensorMap mq, mql, mk2, mv2;
    if (!make_bshd_map_box(&mq, qsrc, s.B, s.Sq, s.H, D, p.group, p.rows_i) ||
        !make_bshd_map_box(&mql, qlo, s.B, s.Sq, s.H, D, p.group, p.rows_i) ||
        !make_bshd_map(&mk2, k, mb, mrows, s.Hk, D, M::TK) || !make_bshd_map(&mv2, v, mb, mrows, s.Hk, D, M::TK))
      return FA_ERR_CUDA;
    const dim3 mgrid(n, s.Hk * p.n_rb, s.B);
    if (rot) {
      using MR = DecMmaCfg<D, D <= 128>;
      auto kr = fa_decode_mma_kernel<D, D <= 128>;
      if (cudaFuncSetAttribute(kr, cudaFuncAttributeMaxDynamicSharedMemorySize, MR::SMEM_BYTES) != cudaSuccess)
        return FA_ERR_CUDA;
      kr<<<mgrid, MR::THREADS, MR::SMEM_BYTES, stream>>>(mq, mql, mk2, mv2, p);
    } else {
      auto kq = fa_decode_mma_kernel<D, false>;
      if (cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, M::SMEM_BYTES) != cudaSuccess)
        return FA_ERR_CUDA;
      kq<<<mgrid, M::THREADS, M::SMEM_BYTES, stream>>>(mq, mql, mk2, mv2, p);
    }
  } else {
    kern<<<dim3(n, s.Hk * p.n_rb, s.B), C::THREADS, C::SMEM_BYTES, stream>>>(mk, mv, p);
  }
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  const long long rows = (long long)s.B * s.Sq * s.H;
  fa_decode_combine_kernel<D><<<unsigned(rows), COMBINE_THREADS, 0, stream>>>(
      p.part_o, p.part_l, static_cast<__nv_bfloat16*>(out), lse, s.Sq, s.H, n);
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
