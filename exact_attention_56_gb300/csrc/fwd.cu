// Forward attention kernel for sm_103a.
//
// Method (page "FlashAttention：快速且内存高效的准确注意力机制", section
// "算法 / 前向传播"): Q is cut into 128-row tiles; for each tile the K/V
// tiles are streamed once; an online softmax keeps an UNSCALED output O and
// the row statistics (m, l), divides O by l only after the last tile, and
// saves the row logsumexp L = m + log l for the backward.
//
// GB300 mapping (one CTA = NT query tiles of 128 rows of one (b, h)):
//   warp 0        TMA producer: Q once, then K_j, V_j into a ring of smem slots
//   warp 1        TMEM allocator and tcgen05.mma issuer (the whole warp runs
//                 the loop, one elected lane issues each MMA):
//                   S_t = Q_t K_j^T  -> TMEM (fp32, 128 columns)
//                   O_t += P_t V_j   -> TMEM (fp32, D columns), P_t read from TMEM
//   warps 4..     one softmax warpgroup per query tile; thread r owns row r of
//                 the tile (TMEM lane r): it reads its S row, applies mask and
//                 ALiBi, updates (m, l), writes P (bf16) back over its S columns,
//                 rescales its O row in TMEM when the running max moved by more
//                 than 2^8, and finally normalises O and writes O and L.
// The MMA order for NT = 2 interleaves the two tiles so each softmax group has
// two MMAs' worth of time per K/V tile. At D = 64 a third S buffer fits in
// TMEM; S of a tile's next K/V tile is then queued while its softmax still
// runs, so each softmax group goes from one K/V tile to the next without
// waiting for its PV and S MMAs.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "../../include/fa.h"
#include "internal.h"
#include "philox.cuh"
#include "ptx.cuh"

namespace fa {

struct FwdParams {
  __nv_bfloat16* out;
  float* lse;
  const float* alibi;
  int alibi_bstride;
  int B, Sq, Sk, H;   // Sq, Sk: padded layout; with cu_q the longest sequences
  int group;          // query heads per key/value head (H / Hk)
  // Packed sequences (page section "代码解读博客：FlashSelfAttention": cu_seqlens):
  // NULL for the padded (B, S, H, D) layout; else device int32 (B + 1,) prefix
  // sums, q/out rows cu_q[b] .. cu_q[b+1]-1 of a (total_q, H, D) tensor and lse
  // (H, total_q).
  const int* cu_q;
  const int* cu_k;
  int total_q;
  Dropout drop;  // used by the DROP instances only
  int wl, wr;
  float scale_log2;  // softmax scale * log2(e)
  unsigned int* status;
  uint64_t wait_ns;      // bounded-wait limit
  unsigned int inject;   // FA_INJECT_* (diagnostics only)
};

template <int D, int NT>
struct FwdCfg {
  static constexpr int PANELS = D / 64;
  static constexpr int PANEL_BYTES = 128 * 128;  // 128 rows x 128 B
  static constexpr int TILE_BYTES = PANELS * PANEL_BYTES;
  // K/V ring. At D = 256 the query tile takes 64 KB, so the ring holds half
  // tiles (two 64-column panels, 32 KB): five of them. A whole-tile ring
  // (two 64 KB slots) made each K and V load wait for the previous tile's
  // MMAs and left its latency on the critical path.
  static constexpr bool HALVES = D == 256;
  static constexpr int SLOT_BYTES = HALVES ? 2 * PANEL_BYTES : TILE_BYTES;
  static constexpr int NSLOT = D == 64 ? 8 : (D == 128 ? 4 : 5);
  static constexpr int THREADS = 128 * (1 + NT);
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = NT * TILE_BYTES;
  static constexpr int BAR_OFF = KV_OFF + NSLOT * SLOT_BYTES;
  static constexpr int SMEM_BYTES = BAR_OFF + 512 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  // S buffers (128 columns each): two, or three where the TMEM budget allows
  // (D = 64, two query tiles). With three, the n-th S tile (n = 2 j + t for
  // key tile j, query tile t) uses buffer n % 3, so S of a query tile's next
  // key tile is issued before that tile's softmax has finished.
  static constexpr int NSB = (NT == 2 && D == 64) ? 3 : 2;
  static constexpr uint32_t O_COL0 = NSB * 128;
  static_assert(NT == 1 || O_COL0 + NT * D <= 512, "TMEM budget");
};

struct FwdBars {
  uint64_t q_full;
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t s_full[3];   // per S buffer
  uint64_t p_full[3];   // per S buffer (P is written over its S)
  uint64_t pv_done[2];  // per query tile
  uint64_t o_done[2];   // per query tile: one phase, after its last PV
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(FwdBars) <= 512, "barrier block");

// Wait-site codes for the status word (kernel 1).
enum : uint32_t {
  SITE_PROD_EMPTY = 0x11,
  SITE_MMA_Q = 0x12,
  SITE_MMA_K = 0x13,
  SITE_MMA_V = 0x14,
  SITE_MMA_P = 0x15,
  SITE_SM_S = 0x16,
  SITE_SM_PV = 0x17,
  SITE_SM_EPI = 0x18,
};

// Stream positions of the half tiles at D = 256 (the producer's order:
// K0lo K0hi | K1lo K1hi V0lo V0hi | ... | V(n-1)lo V(n-1)hi); hi follows lo.
__device__ __forceinline__ int fwd_pos_k(int j) { return j == 0 ? 0 : 4 * j - 2; }
__device__ __forceinline__ int fwd_pos_v(int j, int n_blocks) { return 4 * j + (j + 1 < n_blocks ? 4 : 2); }

// Timeout-only wait used while draining after an abort.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// VARLEN: packed sequences (cu_q, cu_k set); a separate instance, so the padded
// layout keeps its lengths in kernel parameters rather than registers.
// DROP: dropout on the probabilities that multiply V (the row sums use the
// undropped ones, so L is unchanged).
template <int D, int NT, bool VARLEN, bool DROP>
__global__ void __launch_bounds__(FwdCfg<D, NT>::THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = FwdCfg<D, NT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + C::BAR_OFF);

  const int warp = int(warp_id());
  const int lane = int(lane_id());

  // x: rank of this CTA's query group, longest first for right-bounded masks.
  // With 16 or more groups per head the ranks are ordered across the whole
  // grid (block_coord); with fewer, a head's groups stay together, where the
  // balance is already fine and its K/V stays in L2.
  const BlockCoord bc = block_coord(p.wr >= 0 && gridDim.x >= 16);
  const int h = bc.y;
  const int hkv = h / p.group;  // key/value head of this query head
  const int b = bc.z;
  // This sequence's lengths and first rows; tb is the TMA batch coordinate.
  int Sq = p.Sq, Sk = p.Sk, q_off = 0, k_off = 0, tb = b;
  if (VARLEN) {
    q_off = p.cu_q[b];
    Sq = p.cu_q[b + 1] - q_off;
    k_off = p.cu_k[b];
    Sk = p.cu_k[b + 1] - k_off;
    tb = 0;
  }
  const int n_groups = (Sq + NT * 128 - 1) / (NT * 128);
  if (bc.x >= n_groups) return;  // shorter than the longest sequence: no rows here
  // Groups with more live keys first (causal / right-bounded windows).
  const int qg = (p.wr >= 0) ? (n_groups - 1 - bc.x) : bc.x;
  const int row0 = qg * NT * 128;
  const int last_row = min(Sq, row0 + NT * 128) - 1;

  const RowRange first_rr = live_range(row0, Sq, Sk, p.wl, p.wr);
  const RowRange last_rr = live_range(last_row, Sq, Sk, p.wl, p.wr);
  const int kv_lo = first_rr.lo;
  const int kv_hi = last_rr.hi;
  const int jb = kv_lo / 128;
  const int n_blocks = (kv_hi >= kv_lo) ? (kv_hi / 128 + 1 - jb) : 0;
  // Order of the key tiles. ALiBi's bias peaks at each row's diagonal key, so
  // the tile holding the last row's diagonal goes first, then the tiles to its
  // left (falling bias), then those to its right: the running max is set early
  // and O is rarely rescaled. Without ALiBi (jd = 0) the order is ascending.
  const int jd = (p.alibi != nullptr && n_blocks > 0)
                     ? min(max((last_row + Sk - Sq) / 128 - jb, 0), n_blocks - 1)
                     : 0;
  auto key_tile = [jb, jd](int jj) { return jb + (jj <= jd ? jd - jj : jj); };

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int s = 0; s < C::NSB; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->p_full[s], 4);  // one arrive per softmax warp
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->pv_done[s], 1);
      mbar_init(&bars->o_done[s], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
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
      tma_prefetch_desc_w(&tm_k);
      tma_prefetch_desc_w(&tm_v);
      mbar_arrive_expect_tx_w(&bars->q_full, NT * C::TILE_BYTES);
      for (int t = 0; t < NT; ++t)
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d_w(smem + C::Q_OFF + t * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_q, &bars->q_full, pn * 64,
                      h, q_off + row0 + t * 128, tb);
      int issued = 0;
      bool ok = true;
      if constexpr (C::HALVES) {
        // Half tiles in the order the MMAs consume them, K one key tile ahead of
        // V: K0lo K0hi | K1lo K1hi V0lo V0hi | ... | V(n-1)lo V(n-1)hi (stream
        // positions fwd_pos_k / fwd_pos_v); lo holds head dims 0-127, hi 128-255.
        for (int bb = 0; bb <= n_blocks && ok; ++bb) {
          for (int e = 0; e < 4; ++e) {
            const bool isk = e < 2;
            if (isk ? bb >= n_blocks : bb == 0) continue;
            const int j = isk ? bb : bb - 1;
            const int half = e & 1;
            const int s = issued % C::NSLOT;
            const uint32_t ph = uint32_t(issued / C::NSLOT) & 1u;
            if (!fa_wait_warp(&bars->kv_empty[s], ph ^ 1u, watch, SITE_PROD_EMPTY)) {
              ok = false;
              break;
            }
            if (!(p.inject == FA_INJECT_FWD_SKIP_K && isk && j == 1)) {  // diagnostics: key tile 1 never arrives
              mbar_arrive_expect_tx_w(&bars->kv_full[s], C::SLOT_BYTES);
              for (int pl = 0; pl < 2; ++pl)
                tma_load_4d_w(smem + C::KV_OFF + s * C::SLOT_BYTES + pl * C::PANEL_BYTES, isk ? &tm_k : &tm_v,
                              &bars->kv_full[s], (2 * half + pl) * 64, hkv, k_off + key_tile(j) * 128, tb);
            }
            ++issued;
          }
        }
      } else {
        for (int jj = 0; jj < n_blocks && ok; ++jj) {
          for (int kv = 0; kv < 2; ++kv) {
            const int it = 2 * jj + kv;
            const int s = it % C::NSLOT;
            const uint32_t ph = uint32_t(it / C::NSLOT) & 1u;
            if (!fa_wait_warp(&bars->kv_empty[s], ph ^ 1u, watch, SITE_PROD_EMPTY)) {
              ok = false;
              break;
            }
            if (p.inject == FA_INJECT_FWD_SKIP_K && it == 2) {  // diagnostics: key tile 1 never arrives
              issued = it + 1;
              continue;
            }
            mbar_arrive_expect_tx_w(&bars->kv_full[s], C::TILE_BYTES);
            const CUtensorMap* m = kv ? &tm_v : &tm_k;
            for (int pn = 0; pn < C::PANELS; ++pn)
              tma_load_4d_w(smem + C::KV_OFF + s * C::TILE_BYTES + pn * C::PANEL_BYTES, m, &bars->kv_full[s],
                            pn * 64, hkv, k_off + key_tile(jj) * 128, tb);
            issued = it + 1;
          }
        }
      }
      // every copy must land before the CTA may leave (those of an aborted run
      // included; on a normal run the consumers have waited for them already)
      drain_wait(&bars->q_full, 0, p.wait_ns);
      for (int it = (issued > C::NSLOT ? issued - C::NSLOT : 0); it < issued; ++it)
        drain_wait(&bars->kv_full[it % C::NSLOT], uint32_t(it / C::NSLOT) & 1u, p.wait_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop; one elected lane issues each MMA and commit.
    if (n_blocks > 0) {
      constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, 0, 0);  // Q, K both K-major
      constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, 0, 1);    // P from TMEM, V MN-major
      // Descriptors are built once; each k-step, Q tile and ring slot is a
      // constant added to the start-address field, so issuing keeps pace with
      // the tensor pipe.
      const uint64_t q_desc = sdesc_sw128(smem_u32(smem + C::Q_OFF), 16, 1024);
      const uint64_t kv_kdesc = sdesc_sw128(smem_u32(smem + C::KV_OFF), 16, 1024);            // K-major (K)
      const uint64_t kv_mdesc = sdesc_sw128(smem_u32(smem + C::KV_OFF), C::PANEL_BYTES, 1024);  // MN-major (V)

      auto slot_of = [](int it) { return it % C::NSLOT; };
      auto wait_full = [&](int it, uint32_t site) {
        return fa_wait_warp(&bars->kv_full[slot_of(it)], uint32_t(it / C::NSLOT) & 1u, watch, site);
      };
      auto issue_s = [=](int jj, int t, int sbuf) {
        const uint64_t qd = sdesc_adv(q_desc, uint32_t(t) * C::TILE_BYTES);
        const uint64_t kd = sdesc_adv(kv_kdesc, uint32_t(slot_of(2 * jj)) * C::TILE_BYTES);
        const uint32_t ts = tmem + uint32_t(sbuf) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::PANEL_BYTES + (kk % 4) * 32;
          mma_ss_w(ts, sdesc_adv(qd, off), sdesc_adv(kd, off), IDESC_S, kk > 0 ? 1u : 0u);
        }
      };
      // The epilogue waits on o_done, which completes once, after the tile's last
      // PV: pv_done can be more than one phase behind at that point.
      auto last_pv = [&](int jj, int t) {
        if (jj == n_blocks - 1) mma_commit_w(&bars->o_done[t]);
      };
      auto issue_pv = [=](int jj, int t, int sbuf) {
        const uint64_t vd = sdesc_adv(kv_mdesc, uint32_t(slot_of(2 * jj + 1)) * C::TILE_BYTES);
        const uint32_t to = tmem + C::O_COL0 + uint32_t(t) * D, tp = tmem + uint32_t(sbuf) * 128;
        const uint32_t acc0 = jj > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ts_w(to, tp + kk * 8, sdesc_adv(vd, kk * 2048), IDESC_O, kk > 0 ? 1u : acc0);
      };

      bool ok = fa_wait_warp(&bars->q_full, 0, watch, SITE_MMA_Q);
      tc_fence_after();
      if (NT == 2 && C::NSB == 3) {
        // S tile n = 2 jj + t goes to buffer n % 3. Per key tile jj:
        //   PV_0(jj), S_1(jj+1), PV_1(jj), S_0(jj+2).
        // Each S overwrites the buffer whose P the PV just issued has read (in
        // order), and S of a query tile's next key tile is already queued while
        // its softmax runs.
        auto s_tile = [&](int jj, int t) {  // S_t(jj) into its buffer
          const int n = 2 * jj + t;
          issue_s(jj, t, n % 3);
          mma_commit_w(&bars->s_full[n % 3]);
        };
        auto pv_tile = [&](int jj, int t) {  // PV_t(jj) once its P is stored
          const int n = 2 * jj + t;
          if (!fa_wait_warp(&bars->p_full[n % 3], uint32_t(n / 3) & 1u, watch, SITE_MMA_P)) return false;
          tc_fence_after();
          issue_pv(jj, t, n % 3);
          mma_commit_w(&bars->pv_done[t]);
          last_pv(jj, t);
          return true;
        };
        if ((ok = wait_full(0, SITE_MMA_K))) {
          tc_fence_after();
          s_tile(0, 0);
          s_tile(0, 1);
          mma_commit_w(&bars->kv_empty[slot_of(0)]);  // K_0: read by both S tiles
          if (n_blocks > 1 && (ok = wait_full(2, SITE_MMA_K))) {
            tc_fence_after();
            s_tile(1, 0);
          }
        }
        for (int jj = 0; jj < n_blocks && ok; ++jj) {
          if (!(ok = wait_full(2 * jj + 1, SITE_MMA_V))) break;
          if (!(ok = pv_tile(jj, 0))) break;
          if (jj + 1 < n_blocks) {  // K_{jj+1} is already resident (S_0(jj+1) read it)
            s_tile(jj + 1, 1);
            mma_commit_w(&bars->kv_empty[slot_of(2 * (jj + 1))]);
          }
          if (!(ok = pv_tile(jj, 1))) break;
          mma_commit_w(&bars->kv_empty[slot_of(2 * jj + 1)]);  // V_jj: read by both PV tiles
          if (jj + 2 < n_blocks) {
            if (!(ok = wait_full(2 * (jj + 2), SITE_MMA_K))) break;
            tc_fence_after();
            s_tile(jj + 2, 0);
          }
        }
      } else if (NT == 2) {
        for (int jj = 0; jj < n_blocks && ok; ++jj) {
          if (!(ok = wait_full(2 * jj, SITE_MMA_K))) break;
          tc_fence_after();
          issue_s(jj, 0, 0);
          mma_commit_w(&bars->s_full[0]);
          if (jj > 0) {
            if (!(ok = fa_wait_warp(&bars->p_full[1], uint32_t(jj - 1) & 1u, watch, SITE_MMA_P))) break;
            tc_fence_after();
            issue_pv(jj - 1, 1, 1);
            mma_commit_w(&bars->pv_done[1]);
            last_pv(jj - 1, 1);
            mma_commit_w(&bars->kv_empty[slot_of(2 * (jj - 1) + 1)]);
          }
          issue_s(jj, 1, 1);
          mma_commit_w(&bars->s_full[1]);
          mma_commit_w(&bars->kv_empty[slot_of(2 * jj)]);
          if (!(ok = wait_full(2 * jj + 1, SITE_MMA_V))) break;
          if (!(ok = fa_wait_warp(&bars->p_full[0], uint32_t(jj) & 1u, watch, SITE_MMA_P))) break;
          tc_fence_after();
          issue_pv(jj, 0, 0);
          mma_commit_w(&bars->pv_done[0]);
          last_pv(jj, 0);
        }
        if (ok) {
          const int jj = n_blocks - 1;
          if ((ok = fa_wait_warp(&bars->p_full[1], uint32_t(jj) & 1u, watch, SITE_MMA_P))) {
            tc_fence_after();
            issue_pv(jj, 1, 1);
            mma_commit_w(&bars->pv_done[1]);
            last_pv(jj, 1);
            mma_commit_w(&bars->kv_empty[slot_of(2 * jj + 1)]);
          }
        }
      } else if constexpr (C::HALVES) {
        // One query tile, half-tile K/V ring (D = 256). Same order as below:
        // S(jj+1) into the other S buffer, then PV(jj). S takes K in two halves
        // of eight k-steps; PV writes O in two N = 128 halves, each reading its
        // V half. Each half's ring slot is released as soon as its MMAs finish.
        constexpr uint32_t IDESC_O_HALF = idesc_bf16_f32(128, 128, 0, 1);
        auto wait_half = [&](int pos, uint32_t site) {
          return fa_wait_warp(&bars->kv_full[pos % C::NSLOT], uint32_t(pos / C::NSLOT) & 1u, watch, site);
        };
        auto s_halves = [&](int jj, int sbuf) {  // S(jj) = Q K^T into buffer sbuf
          const uint32_t ts = tmem + uint32_t(sbuf) * 128;
          const int pos = fwd_pos_k(jj);
          for (int hh = 0; hh < 2; ++hh) {
            if (!wait_half(pos + hh, SITE_MMA_K)) return false;
            tc_fence_after();
            const uint64_t kd = sdesc_adv(kv_kdesc, uint32_t((pos + hh) % C::NSLOT) * C::SLOT_BYTES);
#pragma unroll
            for (int k8 = 0; k8 < 8; ++k8) {
              const int kk = 8 * hh + k8;
              const uint32_t qoff = (kk / 4) * C::PANEL_BYTES + (kk % 4) * 32;
              const uint32_t koff = (k8 / 4) * C::PANEL_BYTES + (k8 % 4) * 32;
              mma_ss_w(ts, sdesc_adv(q_desc, qoff), sdesc_adv(kd, koff), IDESC_S, kk > 0 ? 1u : 0u);
            }
            mma_commit_w(&bars->kv_empty[(pos + hh) % C::NSLOT]);
          }
          mma_commit_w(&bars->s_full[sbuf]);
          return true;
        };
        auto pv_halves = [&](int jj, int sbuf) {  // O += P V, P in buffer sbuf
          const uint32_t tp = tmem + uint32_t(sbuf) * 128;
          const int pos = fwd_pos_v(jj, n_blocks);
          for (int hh = 0; hh < 2; ++hh) {
            if (!wait_half(pos + hh, SITE_MMA_V)) return false;
            tc_fence_after();
            const uint64_t vd = sdesc_adv(kv_mdesc, uint32_t((pos + hh) % C::NSLOT) * C::SLOT_BYTES);
            const uint32_t to = tmem + C::O_COL0 + uint32_t(hh) * 128;
            const uint32_t acc0 = jj > 0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts_w(to, tp + kk * 8, sdesc_adv(vd, kk * 2048), IDESC_O_HALF, kk > 0 ? 1u : acc0);
            mma_commit_w(&bars->kv_empty[(pos + hh) % C::NSLOT]);
          }
          mma_commit_w(&bars->pv_done[0]);
          last_pv(jj, 0);
          return true;
        };
        ok = ok && s_halves(0, 0);
        for (int jj = 0; jj < n_blocks && ok; ++jj) {
          if (jj + 1 < n_blocks && !(ok = s_halves(jj + 1, (jj + 1) & 1))) break;
          // P barriers per S buffer, as below
          if (!(ok = fa_wait_warp(&bars->p_full[jj & 1], uint32_t(jj >> 1) & 1u, watch, SITE_MMA_P))) break;
          tc_fence_after();
          if (!(ok = pv_halves(jj, jj & 1))) break;
        }
      } else {
        if (ok && (ok = wait_full(0, SITE_MMA_K))) {
          tc_fence_after();
          issue_s(0, 0, 0);
          mma_commit_w(&bars->s_full[0]);
          mma_commit_w(&bars->kv_empty[slot_of(0)]);
        }
        for (int jj = 0; jj < n_blocks && ok; ++jj) {
          if (jj + 1 < n_blocks) {
            if (!(ok = wait_full(2 * (jj + 1), SITE_MMA_K))) break;
            tc_fence_after();
            issue_s(jj + 1, 0, (jj + 1) & 1);
            mma_commit_w(&bars->s_full[(jj + 1) & 1]);
            mma_commit_w(&bars->kv_empty[slot_of(2 * (jj + 1))]);
          }
          if (!(ok = wait_full(2 * jj + 1, SITE_MMA_V))) break;
          // P barriers per S buffer: S(jj+1) is queued before this wait, so the
          // softmax may finish tile jj+1 before it; buffer jj & 1 is next used by
          // S(jj+2), issued after PV(jj)
          if (!(ok = fa_wait_warp(&bars->p_full[jj & 1], uint32_t(jj >> 1) & 1u, watch, SITE_MMA_P))) break;
          tc_fence_after();
          issue_pv(jj, 0, jj & 1);
          mma_commit_w(&bars->pv_done[0]);
          last_pv(jj, 0);
          mma_commit_w(&bars->kv_empty[slot_of(2 * jj + 1)]);
        }
      }
      if (!ok) {  // let issued MMAs finish before TMEM is released
        mma_commit_w(&bars->drain);
        drain_wait(&bars->drain, 0, p.wait_ns);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) / 4;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int i = row0 + t * 128 + r;
    const uint32_t lane_addr = uint32_t(wq * 32) << 16;
    const RowRange rr = live_range(i, Sq, Sk, p.wl, p.wr);
    const int tile_first = row0 + t * 128;
    const int tile_last = min(Sq - 1, tile_first + 127);
    const int tile_lo_max = live_range(tile_last, Sq, Sk, p.wl, p.wr).lo;
    const int tile_hi_min = live_range(tile_first, Sq, Sk, p.wl, p.wr).hi;
    const bool has_alibi = p.alibi != nullptr;
    const float slope_log2 =
        has_alibi ? p.alibi[b * p.alibi_bstride + h] * 1.4426950408889634f : 0.0f;
    const int c_i = i + Sk - Sq;
    const float sl = p.scale_log2;

    float m = -INFINITY;  // reference max (log2 units) the running O and l are relative to
    float l = 0.0f;
    bool ok = true;
    for (int jj = 0; jj < n_blocks; ++jj) {
      // S buffer of this tile and the parity of its use (see FwdCfg::NSB)
      const int n_s = 2 * jj + t;
      const int sb = (C::NSB == 3) ? n_s % 3 : ((NT == 2) ? t : (jj & 1));
      const uint32_t par = (C::NSB == 3) ? (uint32_t(n_s / 3) & 1u)
                                         : ((NT == 2) ? (uint32_t(jj) & 1u) : (uint32_t(jj >> 1) & 1u));
      if (!(ok = fa_wait_warp(&bars->s_full[sb], par, watch, SITE_SM_S))) break;
      tc_fence_after();
      float x[128];
      tmem_ld_x128f(tmem + lane_addr + sb * 128, x);

      const int kbase = key_tile(jj) * 128;
      const bool need_mask = !(kbase >= tile_lo_max && kbase + 127 <= tile_hi_min);
      if (has_alibi) {
        // x = scale*log2(e)*qk - slope*log2(e)*|c(i) - j|, in log2 units
        const float d0 = float(c_i - kbase);
        if (kbase + 127 <= c_i || kbase >= c_i) {
          // All keys on one side of the diagonal: |c(i) - j| = +-(d0 - c), so the
          // bias runs on column pairs. The distances are exact integers and the
          // signed slope times d rounds as -slope * |d| does, so the values are
          // those of the scalar form below.
          const float ns = (kbase >= c_i) ? slope_log2 : -slope_log2;
          const uint64_t ns2 = f2_pack(ns, ns), sl2 = f2_pack(sl, sl), st2 = f2_pack(8.0f, 8.0f);
          uint64_t dist[4];  // four independent chains of column pairs, 8 columns apart
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
      if (need_mask) {
        const int lo = rr.lo - kbase, hi = rr.hi - kbase;
#pragma unroll
        for (int c = 0; c < 128; ++c) x[c] = (c >= lo && c <= hi) ? x[c] : -INFINITY;
      }
      // row max: four independent chains of three-input max over x[0..127]
      float mq[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) mq[k] = fmaxf(x[2 * k], x[2 * k + 1]);
#pragma unroll
      for (int c = 8; c < 128; c += 8) {
#pragma unroll
        for (int k = 0; k < 4; ++k) mq[k] = max3f(mq[k], x[c + 2 * k], x[c + 2 * k + 1]);
      }
      static_assert(8 + 15 * 8 == 128, "max loop covers exactly 128 columns");
      const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      // block max in log2 units (without ALiBi, x still holds raw q.k)
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
      // without ALiBi: p = 2^(x*sl - m); with ALiBi x is already in log2 units.
      // Pairs of columns go through the paired f32x2 FMA and add (each lane
      // rounds exactly as fmaf / + do); rs[k] sums the columns c with
      // c % 4 == k.
      const float mul = has_alibi ? 1.0f : sl;
      const uint64_t mul2 = f2_pack(mul, mul), nm2 = f2_pack(-m_use, -m_use);
      uint64_t rs2[2] = {f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f)};
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t pk[16];
        uint32_t keep = 0;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c = q4 * 32 + 2 * e;
          float a0, a1;
          f2_unpack(f2_fma(f2_pack(x[c], x[c + 1]), mul2, nm2), a0, a1);
          float p0 = ex2_approx(a0);
          float p1 = ex2_approx(a1);
          rs2[e & 1] = f2_add(rs2[e & 1], f2_pack(p0, p1));
          if (DROP) {
            if ((e & 1) == 0) keep = dropout_keep4(p.drop, b * p.H + h, i, (kbase + c) >> 2);
            const int sh = (c & 3);
            p0 = (keep >> sh) & 1u ? p0 * p.drop.keep_scale : 0.0f;
            p1 = (keep >> (sh + 1)) & 1u ? p1 * p.drop.keep_scale : 0.0f;
          }
          pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st_x16(tmem + lane_addr + sb * 128 + q4 * 16, pk);
      }
      float rs[4];
      f2_unpack(rs2[0], rs[0], rs[1]);
      f2_unpack(rs2[1], rs[2], rs[3]);
      l += (rs[0] + rs[1]) + (rs[2] + rs[3]);
      const bool rescale = alpha != 1.0f;
      if (__any_sync(0xffffffffu, rescale) && jj > 0) {
        // O must hold P_{j-1} V_{j-1} before it is rescaled (P_j is already in TMEM).
        if (!(ok = fa_wait_warp(&bars->pv_done[t], uint32_t(jj - 1) & 1u, watch, SITE_SM_PV))) break;
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          const uint32_t oa = tmem + lane_addr + C::O_COL0 + t * D + cc * 32;
          tmem_ld_x32(oa, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st_x32(oa, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(&bars->p_full[(C::NSB == 3 || NT == 1) ? sb : t]);
    }

    // ------------------------------------------------------------ epilogue
    // The sequence's length and first row are read again here rather than kept
    // live across the loop, which would cost registers in the loop.
    const int e_off = VARLEN ? p.cu_q[b] : 0;
    const int e_sq = VARLEN ? p.cu_q[b + 1] - e_off : p.Sq;
    const bool row_ok = i < e_sq;
    const size_t orow = ((VARLEN ? size_t(e_off) + i : size_t(b) * e_sq + i) * p.H + h) * size_t(D);
    const size_t lrow = VARLEN ? size_t(h) * p.total_q + e_off + i : (size_t(b) * p.H + h) * e_sq + i;
    if (n_blocks == 0) {
      if (row_ok) {
        uint4 z = make_uint4(0, 0, 0, 0);
        uint4* dst = reinterpret_cast<uint4*>(p.out + orow);
        for (int e = 0; e < D / 8; ++e) dst[e] = z;
        p.lse[lrow] = -INFINITY;
      }
    } else if (ok && fa_wait_warp(&bars->o_done[t], 0, watch, SITE_SM_EPI)) {
      tc_fence_after();
      const float inv = (l > 0.0f) ? 1.0f / l : 0.0f;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld_x32(tmem + lane_addr + C::O_COL0 + t * D + cc * 32, o);
        if (row_ok) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(p.out + orow + cc * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      }
      if (row_ok)
        p.lse[lrow] = (l > 0.0f) ? (m + lg2_approx(l)) * 0.6931471805599453f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, int NT>
static int launch_fwd_t(const AttnShape& s, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                        void* out, float* lse, const VarlenArgs* vl, const Dropout* dr, cudaStream_t stream) {
  using C = FwdCfg<D, NT>;
  const bool drop = dr && dr->thr != 0;
  if (vl && drop) return FA_ERR_UNSUPPORTED;  // dropout is built for the padded layout
  auto kern = vl ? fa_fwd_kernel<D, NT, true, false>
                 : (drop ? fa_fwd_kernel<D, NT, false, true> : fa_fwd_kernel<D, NT, false, false>);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
    return FA_ERR_CUDA;
  FwdParams p;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.alibi = s.alibi;
  p.alibi_bstride = s.alibi_bstride;
  p.B = s.B;
  p.Sq = s.Sq;
  p.Sk = s.Sk;
  p.H = s.H;
  p.group = s.H / s.Hk;
  p.cu_q = vl ? vl->cu_q : nullptr;
  p.cu_k = vl ? vl->cu_k : nullptr;
  p.total_q = vl ? vl->total_q : 0;
  p.drop = dr ? *dr : Dropout{0, 1.0f, 0, 0, 0};
  p.wl = s.wl;
  p.wr = s.wr;
  p.scale_log2 = s.scale * 1.4426950408889634f;
  p.status = device_status_word();
  {
    const DebugSettings dbg = debug_settings();
    p.wait_ns = dbg.wait_ns;
    p.inject = dbg.inject;
  }
  if (!p.status) return FA_ERR_CUDA;
  dim3 grid((s.Sq + NT * 128 - 1) / (NT * 128), s.H, s.B);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fwd_launch(const AttnShape& s, const void* q, const void* k, const void* v, void* out, float* lse,
               const VarlenArgs* vl, const Dropout* dr, cudaStream_t stream) {
  if (s.B > 65535 || s.H > 65535) return FA_ERR_UNSUPPORTED;
  // Packed sequences are one (1, total, H, D) tensor; s.Sq, s.Sk are then the longest lengths.
  const int mb = vl ? 1 : s.B;
  const int rows_q = vl ? vl->total_q : s.Sq, rows_k = vl ? vl->total_k : s.Sk;
  CUtensorMap mq, mk, mv;
  if (!make_bshd_map(&mq, q, mb, rows_q, s.H, s.D, 128) || !make_bshd_map(&mk, k, mb, rows_k, s.Hk, s.D, 128) ||
      !make_bshd_map(&mv, v, mb, rows_k, s.Hk, s.D, 128))
    return FA_ERR_CUDA;
  switch (s.D) {
    case 64:
      return launch_fwd_t<64, 2>(s, mq, mk, mv, out, lse, vl, dr, stream);
    case 128:
      return launch_fwd_t<128, 2>(s, mq, mk, mv, out, lse, vl, dr, stream);
    case 256:
      return launch_fwd_t<256, 1>(s, mq, mk, mv, out, lse, vl, dr, stream);
    default:
      return FA_ERR_UNSUPPORTED;
  }
}

}  // namespace fa
