// Backward attention kernels for sm_103a.
//
// Method (page "FlashAttention：快速且内存高效的准确注意力机制", sections
// "反向传播" and "并行性 / 反向传播"): only the row logsumexp L is kept from
// the forward; P is recomputed tile by tile from it; the work is parallel over
// key/value column blocks, and dQ is accumulated across blocks by atomic adds.
// Section "2.4" adds a deterministic variant.
//
// Three kernels:
//   fa_bwd_pre      D_i = rowsum(dO_i * O_i), L2_i = L_i*log2(e) (padded to
//                   128-row tiles), zeroes the fp32 dQ accumulator and the
//                   deterministic-mode counters.
//   fa_bwd_main     one CTA per (128-key tile, head, batch); loops over the
//                   live 128-row query tiles:
//                     S^T  = K Q^T                 -> TMEM [0,128)     (tcgen05)
//                     dP^T = V dO^T                -> TMEM [128,256)
//                     P^T  = 2^(S^T*scale*log2e + bias - L2), stored over S^T as
//                            bf16 hi/lo pairs (P = hi + lo to ~2^-16)
//                     dV  += P_hi^T dO + P_lo^T dO (A from TMEM)
//                     dS^T = P^T o (dP^T - D): bf16 hi/lo pairs over dP^T, and
//                            fp16 to shared memory
//                     dK  += dS_hi^T Q + dS_lo^T Q (A from TMEM)
//                     dQ   = dS K in fp16 (K converted once per CTA) -> TMEM [128,128+D)
//                   and drains dQ from TMEM into a swizzled shared-memory stage
//                   (the dS buffer, free once the dQ MMA has read it), from where
//                   TMA bulk reduce-adds it into the fp32 accumulator in L2
//                   (deterministic mode: in key-tile order, behind a counter per
//                   query tile).
//   fa_bwd_convert  dQ = bf16(scale * dQ_acc).
// Precision: the gradients are compared against an fp64 reference with an
// absolute bound close to bf16's own output rounding at |x| ~ 5, so the
// operands of every gradient product carry ~16 significant bits (hi/lo bf16
// pairs or fp16) rather than bf16's 8.
// Warp roles in fa_bwd_main (512 threads): warp 0 TMA producer, warp 1 TMEM
// allocator + MMA issuer, warps 4-11 two compute warpgroups (thread = key row,
// each group one half of the 128 query columns), warps 12-15 dQ warpgroup
// (thread = query row).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "../../include/fa.h"
#include "internal.h"
#include "ptx.cuh"

namespace fa {

struct BwdParams {
  const __nv_bfloat16* dout;
  const __nv_bfloat16* out;
  const float* lse;
  float* dq_acc;   // (B, Sq, H, D) fp32
  float* l2;       // (B, H, Sq_pad): L * log2(e); +inf on rows without keys and on padding
  float* dvec;     // (B, H, Sq_pad): rowsum(dO * O)
  int* sem;        // (B, H, n_qt, 4) ordering counters (deterministic mode)
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const float* alibi;
  int alibi_bstride;
  int B, Sq, Sk, H, Sq_pad, n_qt;
  int wl, wr;
  float scale;
  float scale_log2;
  int deterministic;
  unsigned int* status;
};

template <int D>
struct BwdCfg {
  static constexpr int PANELS = D / 64;
  static constexpr int PANEL_BYTES = 128 * 128;
  static constexpr int TILE_BYTES = PANELS * PANEL_BYTES;
  static constexpr int NQ = 2;                  // Q (+ L2, D) stages
  static constexpr int NDO = D == 64 ? 2 : 1;   // dO stages
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = TILE_BYTES;
  static constexpr int K16_OFF = 2 * TILE_BYTES;  // fp16 copy of K for the dQ product
  static constexpr int Q_OFF = 3 * TILE_BYTES;
  static constexpr int DO_OFF = Q_OFF + NQ * TILE_BYTES;
  static constexpr int DS_OFF = DO_OFF + NDO * TILE_BYTES;  // 128 keys x 128 queries fp16, two 64-query panels
  static constexpr int VEC_OFF = DS_OFF + 2 * PANEL_BYTES;  // per Q stage: L2[128], D[128]
  static constexpr int BAR_OFF = VEC_OFF + NQ * 1024;
  static constexpr int SMEM_BYTES = BAR_OFF + 256;
  static constexpr int THREADS = 512;
  static constexpr int Q_TX = TILE_BYTES + 1024;
  static constexpr uint32_t T_S = 0, T_DP = 128, T_DQ = 128, T_DV = 256, T_DK = 256 + D;
  static_assert(T_DK + D <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct BwdBars {
  uint64_t kv_full;
  uint64_t q_full[2], q_empty[2];
  uint64_t do_full[2], do_empty[2];
  uint64_t s_full, dp_full, p_ready, ds_ready, dq_full, dq_free, acc_done, drain;
  uint64_t staged[2], half_free[2], stage_done;
  uint32_t tmem_base;
  int abort;
};

enum : uint32_t {
  SITE_B_EMPTY = 0x31,
  SITE_B_KV = 0x32,
  SITE_B_FULL = 0x33,
  SITE_B_DQFREE = 0x34,
  SITE_B_P = 0x35,
  SITE_B_DS = 0x36,
  SITE_B_S = 0x37,
  SITE_B_DP = 0x38,
  SITE_B_DQ = 0x39,
  SITE_B_ACC = 0x3A,
  SITE_B_SEM = 0x3B,
  SITE_B_ALIGN = 0x3C,
  SITE_B_DOEMPTY = 0x3D,
  SITE_B_DOFULL = 0x3E,
  SITE_B_STAGE = 0x3F,
};

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void drain_wait_b(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > FA_WAIT_TIMEOUT_NS) return;
  }
}

// Does query tile qt meet key tile kt (does the bounding interval of its rows'
// live keys intersect the key tile)?
__device__ __forceinline__ bool qtile_meets(int qt, int kt, const BwdParams& p) {
  const int r0 = qt * 128;
  const int r1 = min(p.Sq, r0 + 128) - 1;
  const int lo = live_range(r0, p.Sq, p.Sk, p.wl, p.wr).lo;
  const int hi = live_range(r1, p.Sq, p.Sk, p.wl, p.wr).hi;
  if (hi < lo) return false;
  return !(hi < kt * 128 || lo > kt * 128 + 127);
}
// First key tile that meets query tile qt (its rank base for deterministic ordering).
__device__ __forceinline__ int first_ktile(int qt, const BwdParams& p) {
  return live_range(qt * 128, p.Sq, p.Sk, p.wl, p.wr).lo / 128;
}

template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    fa_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // the swizzled layouts need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(p.status, FA_DEV_TIMEOUT | SITE_B_ALIGN);
    return;
  }
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::BAR_OFF);
  const int warp = int(warp_id());
  const int lane = int(lane_id());
  const int kt = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int j0 = kt * 128;

  // Live query tiles of this key tile: a contiguous range.
  const int n_qt = p.n_qt;
  int qt_first = n_qt, qt_last = -1;
  for (int qt = 0; qt < n_qt; ++qt) {
    if (qtile_meets(qt, kt, p)) {
      qt_first = min(qt_first, qt);
      qt_last = qt;
    }
  }
  const int n_iter = qt_last >= qt_first ? qt_last - qt_first + 1 : 0;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
      mbar_init(&bars->do_full[s], 1);
      mbar_init(&bars->do_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_ready, 256);
    mbar_init(&bars->ds_ready, 256);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, 128);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->drain, 1);
    for (int hh = 0; hh < 2; ++hh) {
      mbar_init(&bars->staged[hh], 128);
      mbar_init(&bars->half_free[hh], 1);
    }
    mbar_init(&bars->stage_done, 1);
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
  const Watch watch{&bars->abort, p.status};
  const size_t vec_base = (size_t(b) * p.H + h) * p.Sq_pad;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_iter > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(&bars->kv_full, 2 * C::TILE_BYTES);
      for (int pn = 0; pn < C::PANELS; ++pn) {
        tma_load_4d(smem + C::K_OFF + pn * C::PANEL_BYTES, &tm_k, &bars->kv_full, pn * 64, h, j0, b);
        tma_load_4d(smem + C::V_OFF + pn * C::PANEL_BYTES, &tm_v, &bars->kv_full, pn * 64, h, j0, b);
      }
      int q_issued = 0, do_issued = 0;
      for (int ii = 0; ii < n_iter; ++ii) {
        const int s = ii % C::NQ;
        const int i0 = (qt_first + ii) * 128;
        if (!fa_wait(&bars->q_empty[s], (uint32_t(ii / C::NQ) & 1u) ^ 1u, watch, SITE_B_EMPTY)) break;
        mbar_arrive_expect_tx(&bars->q_full[s], C::Q_TX);
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d(smem + C::Q_OFF + s * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_q, &bars->q_full[s], pn * 64,
                      h, i0, b);
        bulk_load(smem + C::VEC_OFF + s * 1024, p.l2 + vec_base + i0, 512, &bars->q_full[s]);
        bulk_load(smem + C::VEC_OFF + s * 1024 + 512, p.dvec + vec_base + i0, 512, &bars->q_full[s]);
        q_issued = ii + 1;
        const int d = ii % C::NDO;
        if (!fa_wait(&bars->do_empty[d], (uint32_t(ii / C::NDO) & 1u) ^ 1u, watch, SITE_B_DOEMPTY)) break;
        mbar_arrive_expect_tx(&bars->do_full[d], C::TILE_BYTES);
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d(smem + C::DO_OFF + d * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_do, &bars->do_full[d],
                      pn * 64, h, i0, b);
        do_issued = ii + 1;
      }
      // every copy must land before the CTA may exit
      drain_wait_b(&bars->kv_full, 0);
      for (int ii = (q_issued > C::NQ ? q_issued - C::NQ : 0); ii < q_issued; ++ii)
        drain_wait_b(&bars->q_full[ii % C::NQ], uint32_t(ii / C::NQ) & 1u);
      for (int ii = (do_issued > C::NDO ? do_issued - C::NDO : 0); ii < do_issued; ++ii)
        drain_wait_b(&bars->do_full[ii % C::NDO], uint32_t(ii / C::NDO) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t ID_SS = idesc_bf16_f32(128, 128, 0, 0);  // S^T, dP^T: both operands K-major
      constexpr uint32_t ID_TN = idesc_bf16_f32(128, D, 0, 1);    // dV, dK: A from TMEM, B (dO / Q) MN-major
      constexpr uint32_t ID_DQ = idesc_f16_f32(128, D, 1, 1);     // dQ: fp16 A (dS) and B (K), MN-major
      const uint32_t k_a = smem_u32(smem + C::K_OFF);
      const uint32_t v_a = smem_u32(smem + C::V_OFF);
      const uint32_t k16_a = smem_u32(smem + C::K16_OFF);
      const uint32_t ds_a = smem_u32(smem + C::DS_OFF);
      bool ok = fa_wait(&bars->kv_full, 0, watch, SITE_B_KV);
      for (int ii = 0; ii < n_iter && ok; ++ii) {
        const int s = ii % C::NQ;
        const int d = ii % C::NDO;
        const uint32_t q_a = smem_u32(smem + C::Q_OFF + s * C::TILE_BYTES);
        const uint32_t do_a = smem_u32(smem + C::DO_OFF + d * C::TILE_BYTES);
        if (!(ok = fa_wait(&bars->q_full[s], uint32_t(ii / C::NQ) & 1u, watch, SITE_B_FULL))) break;
        tc_fence_after();
        // S^T = K Q^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::PANEL_BYTES + (kk % 4) * 32;
          mma_ss(tmem + C::T_S, sdesc_sw128(k_a + off, 16, 1024), sdesc_sw128(q_a + off, 16, 1024), ID_SS,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->s_full);
        // dP^T = V dO^T, into the columns dQ of the previous tile occupied
        if (ii > 0) {
          if (!(ok = fa_wait(&bars->dq_free, uint32_t(ii - 1) & 1u, watch, SITE_B_DQFREE))) break;
        }
        if (!(ok = fa_wait(&bars->do_full[d], uint32_t(ii / C::NDO) & 1u, watch, SITE_B_DOFULL))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::PANEL_BYTES + (kk % 4) * 32;
          mma_ss(tmem + C::T_DP, sdesc_sw128(v_a + off, 16, 1024), sdesc_sw128(do_a + off, 16, 1024), ID_SS,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->dp_full);
        // dV += P_hi^T dO + P_lo^T dO ; queries 16kk.. sit at column 64*(kk/4) + 16*(kk%4) (hi), +8 (lo)
        if (!(ok = fa_wait(&bars->p_ready, uint32_t(ii) & 1u, watch, SITE_B_P))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t pa = tmem + C::T_S + (kk / 4) * 64 + (kk % 4) * 16;
          const uint64_t bd = sdesc_sw128(do_a + kk * 2048, C::PANEL_BYTES, 1024);
          mma_ts(tmem + C::T_DV, pa, bd, ID_TN, (ii > 0 || kk > 0) ? 1u : 0u);
          mma_ts(tmem + C::T_DV, pa + 8, bd, ID_TN, 1u);
        }
        mma_commit(&bars->do_empty[d]);
        // dK += dS_hi^T Q + dS_lo^T Q ; dQ = dS K (fp16)
        if (!(ok = fa_wait(&bars->ds_ready, uint32_t(ii) & 1u, watch, SITE_B_DS))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t da = tmem + C::T_DP + (kk / 4) * 64 + (kk % 4) * 16;
          const uint64_t bd = sdesc_sw128(q_a + kk * 2048, C::PANEL_BYTES, 1024);
          mma_ts(tmem + C::T_DK, da, bd, ID_TN, (ii > 0 || kk > 0) ? 1u : 0u);
          mma_ts(tmem + C::T_DK, da + 8, bd, ID_TN, 1u);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + C::T_DQ, sdesc_sw128(ds_a + kk * 2048, C::PANEL_BYTES, 1024),
                 sdesc_sw128(k16_a + kk * 2048, C::PANEL_BYTES, 1024), ID_DQ, kk > 0 ? 1u : 0u);
        mma_commit(&bars->dq_full);
        mma_commit(&bars->q_empty[s]);
      }
      if (ok) {
        mma_commit(&bars->acc_done);
      } else {
        mma_commit(&bars->drain);
        drain_wait_b(&bars->drain, 0);
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ compute (thread = key row)
    const int w = (warp - 4) / 4;  // query-column half
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int j = j0 + r;
    const uint32_t lane_addr = uint32_t(wq * 32) << 16;
    const int off = p.Sk - p.Sq;
    // live queries of key j: i in [qlo, qhi]
    auto qbounds = [&](int jj, int& lo, int& hi) {
      lo = (p.wr >= 0) ? jj - off - p.wr : 0;
      hi = (p.wl >= 0) ? jj - off + p.wl : p.Sq - 1;
      lo = max(lo, 0);
      hi = min(hi, p.Sq - 1);
      if (jj >= p.Sk) {
        lo = 1;
        hi = 0;
      }
    };
    int qlo, qhi;
    qbounds(j, qlo, qhi);
    int qlo_max, dummy, qhi_min;
    qbounds(min(p.Sk - 1, j0 + 127), qlo_max, dummy);
    qbounds(j0, dummy, qhi_min);
    const bool tile_keys_ok = j0 + 127 < p.Sk;
    const bool has_alibi = p.alibi != nullptr;
    const float slope_log2 = has_alibi ? p.alibi[b * p.alibi_bstride + h] * 1.4426950408889634f : 0.0f;
    const float sl = p.scale_log2;
    bool ok = true;
    // fp16 copy of K for the dQ product: same swizzled byte layout, element by element.
    if (n_iter > 0) {
      ok = fa_wait_warp(&bars->kv_full, 0, watch, SITE_B_KV);
      if (ok) {
        constexpr int CHUNKS = C::PANELS * 8;  // 16-byte chunks per K row
        const uint8_t* src = smem + C::K_OFF;
        uint8_t* dst = smem + C::K16_OFF;
#pragma unroll
        for (int cidx = w * (CHUNKS / 2); cidx < (w + 1) * (CHUNKS / 2); ++cidx) {
          const int off = (cidx / 8) * C::PANEL_BYTES + r * 128 + (cidx % 8) * 16;
          const uint4 u = *reinterpret_cast<const uint4*>(src + off);
          const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o[e] = pack_f16x2(__uint_as_float(wv[e] << 16), __uint_as_float(wv[e] & 0xFFFF0000u));
          *reinterpret_cast<uint4*>(dst + off) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async_smem();
      }
    }
    for (int ii = 0; ii < n_iter && ok; ++ii) {
      const int s = ii % C::NQ;
      const int i0 = (qt_first + ii) * 128;
      const int ib = i0 + w * 64;  // first query of this half
      const float4* l2v = reinterpret_cast<const float4*>(smem + C::VEC_OFF + s * 1024) + w * 16;
      const float4* dvv = l2v + 32;
      if (!(ok = fa_wait_warp(&bars->s_full, uint32_t(ii) & 1u, watch, SITE_B_S))) break;
      tc_fence_after();
      {
        float pv[64];
        tmem_ld_x64f(tmem + lane_addr + C::T_S + w * 64, pv);
        const bool need_mask = !(tile_keys_ok && i0 >= qlo_max && i0 + 127 <= qhi_min);
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 l4 = l2v[c4];
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 4 * c4 + e;
            float bias = -lv[e];
            if (has_alibi) bias -= slope_log2 * fabsf(float(ib + off - j + c));
            pv[c] = ex2_approx(fmaf(pv[c], sl, bias));
          }
        }
        if (need_mask) {
          const int lo = qlo - ib, hi = qhi - ib;
#pragma unroll
          for (int c = 0; c < 64; ++c) pv[c] = (c >= lo && c <= hi) ? pv[c] : 0.0f;
        }
        // P as bf16 hi/lo pairs; 16-query chunk c4 -> columns [16*c4, 16*c4+8) hi, [+8, +16) lo
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t hl[16];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float a0 = pv[16 * c4 + 2 * e], a1 = pv[16 * c4 + 2 * e + 1];
            const uint32_t hp = pack_bf16x2(a0, a1);
            hl[e] = hp;
            hl[8 + e] = pack_bf16x2(a0 - __uint_as_float(hp << 16), a1 - __uint_as_float(hp & 0xFFFF0000u));
          }
          tmem_st_x16(tmem + lane_addr + C::T_S + w * 64 + 16 * c4, hl);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_ready);

      if (!(ok = fa_wait_warp(&bars->dp_full, uint32_t(ii) & 1u, watch, SITE_B_DP))) break;
      // the dS buffer doubles as the previous tile's dQ stage: wait until TMA has read it
      if (ii > 0 && !(ok = fa_wait_warp(&bars->stage_done, uint32_t(ii - 1) & 1u, watch, SITE_B_STAGE))) break;
      tc_fence_after();
      uint8_t* ds_row = smem + C::DS_OFF + w * C::PANEL_BYTES + r * 128;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float dp[16];
        uint32_t ph[16];  // P hi (8) then lo (8) for these 16 queries
        tmem_ld_x16f(tmem + lane_addr + C::T_DP + w * 64 + 16 * c4, dp);
        tmem_ld_x16(tmem + lane_addr + C::T_S + w * 64 + 16 * c4, ph);
        uint32_t hl[16];
        uint32_t h16[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = 16 * c4 + 2 * e;
          const float4 d4 = dvv[c / 4];
          const float dv0 = (c % 4 == 0) ? d4.x : d4.z;
          const float dv1 = (c % 4 == 0) ? d4.y : d4.w;
          const float p0 = __uint_as_float(ph[e] << 16) + __uint_as_float(ph[8 + e] << 16);
          const float p1 = __uint_as_float(ph[e] & 0xFFFF0000u) + __uint_as_float(ph[8 + e] & 0xFFFF0000u);
          const float s0 = p0 * (dp[2 * e] - dv0);
          const float s1 = p1 * (dp[2 * e + 1] - dv1);
          const uint32_t hp = pack_bf16x2(s0, s1);
          hl[e] = hp;
          hl[8 + e] = pack_bf16x2(s0 - __uint_as_float(hp << 16), s1 - __uint_as_float(hp & 0xFFFF0000u));
          h16[e] = pack_f16x2(s0, s1);
        }
        // dS^T hi/lo over this chunk's own (already read) dP^T columns
        tmem_st_x16(tmem + lane_addr + C::T_DP + w * 64 + 16 * c4, hl);
        // fp16 dS for the dQ product: 16 queries = two 16-byte chunks of row r
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int chunk = (2 * c4 + e) ^ (r & 7);
          *reinterpret_cast<uint4*>(ds_row + chunk * 16) =
              make_uint4(h16[4 * e], h16[4 * e + 1], h16[4 * e + 2], h16[4 * e + 3]);
        }
      }
      fence_proxy_async_smem();
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->ds_ready);
    }
    // ------------------------------------------------------------ dK / dV epilogue
    const bool row_ok = j < p.Sk;
    __nv_bfloat16* dst = (w == 0 ? p.dv : p.dk) + ((size_t(b) * p.Sk + size_t(j)) * p.H + h) * size_t(D);
    const float mul = (w == 0) ? 1.0f : p.scale;
    if (n_iter == 0) {
      if (row_ok)
        for (int e = 0; e < D / 8; ++e) reinterpret_cast<uint4*>(dst)[e] = make_uint4(0, 0, 0, 0);
    } else if (ok && fa_wait_warp(&bars->acc_done, 0, watch, SITE_B_ACC)) {
      tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        float a[32];
        tmem_ld_x32f(tmem + lane_addr + (w == 0 ? C::T_DV : C::T_DK) + cc * 32, a);
        if (row_ok) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(a[2 * e] * mul, a[2 * e + 1] * mul);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            reinterpret_cast<uint4*>(dst + cc * 32)[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ dQ drain (thread = query row)
    // TMEM -> shared stage (two 16 KB halves of 128 rows x 32 fp32, 128-byte
    // swizzle, in the dS buffer) -> TMA reduce-add into dQ_acc. Thread r == 0
    // issues the bulk operations; the handshakes are bounded mbarrier waits.
    constexpr int NCH = D / 32;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_addr = uint32_t(wq * 32) << 16;
    uint8_t* stage = smem + C::DS_OFF;
    uint32_t staged_ph[2] = {0u, 0u};
    for (int ii = 0; ii < n_iter; ++ii) {
      const int qt = qt_first + ii;
      if (!fa_wait_warp(&bars->dq_full, uint32_t(ii) & 1u, watch, SITE_B_DQ)) break;
      tc_fence_after();
      bool ok = true;
#pragma unroll 1
      for (int cc = 0; cc < NCH && ok; ++cc) {
        const int hh = cc & 1;
        if (cc >= 2 && !(ok = fa_wait_warp(&bars->half_free[hh], uint32_t(ii) & 1u, watch, SITE_B_STAGE))) break;
        float a[32];
        tmem_ld_x32f(tmem + lane_addr + C::T_DQ + cc * 32, a);
        uint8_t* row = stage + hh * C::PANEL_BYTES + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<float4*>(row + ((c ^ (r & 7)) << 4)) =
              make_float4(a[4 * c], a[4 * c + 1], a[4 * c + 2], a[4 * c + 3]);
        if (cc == NCH - 1) {  // TMEM fully read: the next dP^T may overwrite it
          tc_fence_before();
          mbar_arrive(&bars->dq_free);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars->staged[hh]);
        if (r == 0) {
          ok = fa_wait(&bars->staged[hh], staged_ph[hh], watch, SITE_B_STAGE);
          if (ok && p.deterministic && cc == 0) {
            // wait for every earlier key tile of this query tile to have finished its adds
            int* sem = p.sem + ((size_t(b) * p.H + h) * p.n_qt + qt) * 4;
            const int rank = kt - first_ktile(qt, p);
            const uint64_t t0 = globaltimer_ns();
            int v;
            for (;;) {
              asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(sem) : "memory");
              if (v == rank) break;
              if (*watch.abort || globaltimer_ns() - t0 > FA_WAIT_TIMEOUT_NS) {
                *watch.abort = 1;
                atomicOr(p.status, FA_DEV_TIMEOUT | SITE_B_SEM);
                ok = false;
                break;
              }
            }
          }
          if (ok) {
            tma_reduce_add_4d(&tm_dq, stage + hh * C::PANEL_BYTES, cc * 32, h, qt * 128, b);
            bulk_commit_group();
            if (cc >= 1 && cc + 1 < NCH) {  // chunk cc-1 read out: its half is free for chunk cc+1
              bulk_wait_group_read<1>();
              mbar_arrive(&bars->half_free[(cc - 1) & 1]);
            }
          }
        }
        staged_ph[hh] ^= 1u;
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0 && !*watch.abort;
      }
      if (!ok) break;
      if (r == 0) {
        bulk_wait_group_read<0>();
        if (p.deterministic) {
          bulk_wait_group<0>();
          __threadfence();
          int* sem = p.sem + ((size_t(b) * p.H + h) * p.n_qt + qt) * 4;
          asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(sem) : "memory");
        }
        mbar_arrive(&bars->stage_done);
      }
      __syncwarp();
    }
    if (lane == 0) bulk_wait_group<0>();  // no bulk operation may outlive the CTA
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// D_i = rowsum(dO * O), L2 = L*log2(e) (+inf where L = -inf or on padding),
// dQ accumulator rows zeroed, counters zeroed. One warp per (b, h, row).
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const BwdParams p) {
  constexpr int PER = D / 32;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  if (blockIdx.x == 0 && p.deterministic)
    for (int t = threadIdx.x; t < p.n_qt * 4; t += blockDim.x) p.sem[(size_t(b) * p.H + h) * p.n_qt * 4 + t] = 0;
  if (row >= p.Sq_pad) return;
  const size_t vi = (size_t(b) * p.H + h) * p.Sq_pad + row;
  if (row >= p.Sq) {
    if (lane == 0) {
      p.dvec[vi] = 0.0f;
      p.l2[vi] = INFINITY;
    }
    return;
  }
  const size_t ro = ((size_t(b) * p.Sq + row) * p.H + h) * size_t(D) + lane * PER;
  float acc = 0.0f;
#pragma unroll
  for (int e = 0; e < PER; e += 2) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(p.dout + ro + e);
    const __nv_bfloat162 o = *reinterpret_cast<const __nv_bfloat162*>(p.out + ro + e);
    acc = fmaf(__low2float(a), __low2float(o), acc);
    acc = fmaf(__high2float(a), __high2float(o), acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
#pragma unroll
  for (int e = 0; e < PER; e += 2) *reinterpret_cast<float2*>(p.dq_acc + ro + e) = make_float2(0.0f, 0.0f);
  if (lane == 0) {
    p.dvec[vi] = acc;
    const float L = p.lse[(size_t(b) * p.H + h) * p.Sq + row];
    p.l2[vi] = (L == -INFINITY) ? INFINITY : L * 1.4426950408889634f;
  }
}

__global__ void __launch_bounds__(256) fa_bwd_convert_kernel(const float* __restrict__ acc,
                                                              __nv_bfloat16* __restrict__ dq, size_t n8,
                                                              float scale) {
  for (size_t t = blockIdx.x * size_t(blockDim.x) + threadIdx.x; t < n8; t += size_t(gridDim.x) * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * t];
    const float4 c = reinterpret_cast<const float4*>(acc)[2 * t + 1];
    reinterpret_cast<uint4*>(dq)[t] = make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                                                 pack_bf16x2(c.x * scale, c.y * scale), pack_bf16x2(c.z * scale, c.w * scale));
  }
}

static size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

size_t bwd_workspace_bytes(int B, int Sq, int Sk, int H, int D, int deterministic) {
  (void)Sk;
  const size_t sq_pad = size_t((Sq + 127) / 128) * 128;
  const size_t n_qt = sq_pad / 128;
  size_t n = al256(size_t(B) * Sq * H * D * 4);  // dQ accumulator
  n += 2 * al256(size_t(B) * H * sq_pad * 4);    // L2, D
  if (deterministic) n += al256(size_t(B) * H * n_qt * 4 * 4);
  return n;
}

template <int D>
static int launch_bwd_t(const AttnShape& s, const void* dout, const void* q, const void* k, const void* v,
                        const void* out, const float* lse, void* dq, void* dk, void* dv, void* ws,
                        int deterministic, cudaStream_t stream) {
  using C = BwdCfg<D>;
  CUtensorMap mq, mk, mv, mdo;
  if (!make_bshd_map(&mq, q, s.B, s.Sq, s.H, D, 128) || !make_bshd_map(&mk, k, s.B, s.Sk, s.H, D, 128) ||
      !make_bshd_map(&mv, v, s.B, s.Sk, s.H, D, 128) || !make_bshd_map(&mdo, dout, s.B, s.Sq, s.H, D, 128))
    return FA_ERR_CUDA;
  BwdParams p;
  p.B = s.B;
  p.Sq = s.Sq;
  p.Sk = s.Sk;
  p.H = s.H;
  p.Sq_pad = ((s.Sq + 127) / 128) * 128;
  p.n_qt = p.Sq_pad / 128;
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.dq_acc = reinterpret_cast<float*>(w);
  w += al256(size_t(s.B) * s.Sq * s.H * D * 4);
  p.l2 = reinterpret_cast<float*>(w);
  w += al256(size_t(s.B) * s.H * p.Sq_pad * 4);
  p.dvec = reinterpret_cast<float*>(w);
  w += al256(size_t(s.B) * s.H * p.Sq_pad * 4);
  p.sem = deterministic ? reinterpret_cast<int*>(w) : nullptr;
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.out = static_cast<const __nv_bfloat16*>(out);
  p.lse = lse;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.alibi = s.alibi;
  p.alibi_bstride = s.alibi_bstride;
  p.wl = s.wl;
  p.wr = s.wr;
  p.scale = s.scale;
  p.scale_log2 = s.scale * 1.4426950408889634f;
  p.deterministic = deterministic ? 1 : 0;
  p.status = device_status_word();
  if (!p.status) return FA_ERR_CUDA;
  if (s.B > 65535 || s.H > 65535) return FA_ERR_UNSUPPORTED;

  fa_bwd_pre_kernel<D><<<dim3(p.Sq_pad / 8, s.H, s.B), 256, 0, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  auto kern = fa_bwd_main_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
    return FA_ERR_CUDA;
  CUtensorMap mdq;
  if (!make_bshd_f32_map(&mdq, p.dq_acc, s.B, s.Sq, s.H, D)) return FA_ERR_CUDA;
  kern<<<dim3((s.Sk + 127) / 128, s.H, s.B), C::THREADS, C::SMEM_BYTES, stream>>>(mq, mk, mv, mdo, mdq, p);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  const size_t n8 = size_t(s.B) * s.Sq * s.H * D / 8;
  size_t nb = (n8 + 255) / 256;
  const size_t cap = size_t(device_sm_count()) * 8;
  if (nb > cap) nb = cap;
  if (nb < 1) nb = 1;
  const int blocks = int(nb);
  fa_bwd_convert_kernel<<<blocks, 256, 0, stream>>>(p.dq_acc, p.dq, n8, s.scale);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int bwd_launch(const AttnShape& s, const void* dout, const void* q, const void* k, const void* v, const void* out,
               const float* lse, void* dq, void* dk, void* dv, void* workspace, int deterministic,
               cudaStream_t stream) {
  switch (s.D) {
    case 64:
      return launch_bwd_t<64>(s, dout, q, k, v, out, lse, dq, dk, dv, workspace, deterministic, stream);
    case 128:
      return launch_bwd_t<128>(s, dout, q, k, v, out, lse, dq, dk, dv, workspace, deterministic, stream);
    default:
      return FA_ERR_UNSUPPORTED;
  }
}

}  // namespace fa
