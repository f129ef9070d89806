// Backward attention kernels for sm_103a.
//
// Method (page "FlashAttention：快速且内存高效的准确注意力机制", sections
// "反向传播" and "并行性 / 反向传播"): only the row logsumexp L is kept from
// the forward and P is recomputed tile by tile from it. Section "2.4" asks
// for a deterministic variant.
//
// The page's own design parallelises over key/value column blocks and adds
// dQ across blocks with atomics. On GB300 per-thread fp32 reductions reach
// about 3 TB/s of adds and bulk tensor reductions about 6 TB/s, against 4.3 GB
// of dQ shares at D = 64 for a 16k-token, 2048-wide sweep point. So the
// reproducible path (deterministic) never reduces across CTAs, and only the
// D = 64 default path adds dQ across key tiles (FDQ below):
//
//   fa_bwd_pre       D_i = rowsum(dO_i * O_i) and L2_i = L_i*log2(e), padded to
//                    128-row tiles (+inf on padding and on rows without keys),
//                    fp16 copies of Q, K, V and dO, and each (sequence,
//                    key/value head) group's largest |q|, |k|, |v|, |dO|.
//   fa_bwd_rescale   copies again, times a power of two, the groups whose
//                    magnitudes lie outside what fp16 keeps exactly (see
//                    "operand range" below); nothing else for the rest.
//   fa_bwd_dkdv      one CTA per (128-key tile, key/value head, batch), looping
//                    over the live 128-row query tiles of every query head
//                    that shares the key/value head:
//                      S^T  = K Q^T                 -> TMEM S region   (tcgen05)
//                      dP^T = V dO^T                -> TMEM dP region
//                      P^T  = 2^(S^T*scale*log2e + bias - L2)
//                      dS^T = P^T o (dP^T - D)      -> both fp16, over dP^T
//                      dV  += P^T dO, dK += dS^T Q  (A from TMEM, two chains)
//                    S^T of the next tile is computed while this one's
//                    exponentials run; then dK (times scale) and dV are written.
//   fa_bwd_dq        one CTA per (128-row query tile, head, batch), looping over
//                    the live key tiles (the forward's shape, thread = query row):
//                      S  = Q K^T -> TMEM, P = 2^(S*scale*log2e + bias - L2)
//                      dP = dO V^T, dS = P o (dP - D) -> fp16 over dP
//                      dQ += dS K
//                    S of the next key tile is computed while this one's
//                    exponentials run; then dQ (times scale) is written once.
// Every output element is produced by one CTA in a fixed order, so every run
// of this path is bitwise reproducible.
//   FDQ (D = 64, deterministic == 0, dense, no dropout): fa_bwd_dkdv also forms
//                    dQ_t = dS K (M = queries) per query tile and adds it into
//                    an fp32 accumulator with TMA reductions; a conversion to
//                    bf16 replaces fa_bwd_dq, whose S and dP are not recomputed.
//
// Precision and MMA rate: every product takes fp16 operands (P, dS and exact
// fp16 copies of the bf16 inputs, scaled per group by a power of two). fp16
// keeps 11 significant bits, enough for the gradients to stay at bf16's own
// output rounding against an fp64 reference with one MMA per product.
//
// Both main kernels follow one schedule: the score tile of the next step is
// issued as soon as the compute warps hold the current one in registers, and
// the operand rings are deep enough that a tile is loaded about one step
// before the MMA that reads it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "../../include/fa.h"
#include "internal.h"
#include "philox.cuh"
#include "ptx.cuh"

namespace fa {

struct BwdParams {
  const __nv_bfloat16* dout;
  const __nv_bfloat16* out;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* lse;
  float* nl2;     // (B, H, Sq_pad): -L * log2(e), the exponent's bias; -inf on rows without keys and on padding
  float* dvec;    // (B, H, Sq_pad): rowsum(dO * O)
  uint16_t* q16;  // fp16 copies, (B, S, H, D) like the inputs
  uint16_t* do16;
  uint16_t* k16;
  uint16_t* v16;
  // (B, Hk, 4) uint32: largest |x| of q, k, v, dout over each (sequence,
  // key/value head) group, as bf16 magnitude bits; see group_exps()
  uint32_t* amax;
  // (B, Hk, AMAX_REPS, 4) uint32: the same maxima as the pre-pass gathers them,
  // spread over replicas so that concurrent atomics rarely share an address
  uint32_t* amax_rep;
  int n_chunks;  // 64-token chunks per sequence (rescale pass)
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const float* alibi;
  int alibi_bstride;
  int B, Sq, Sk, H, Sq_pad, n_qt;  // with cu_q: Sq, Sk the longest sequences
  int Hk, group;  // key/value heads; query heads per key/value head
  // Packed sequences: NULL for the padded layout, else device int32 (B + 1,)
  // prefix sums into (total_q, H, D) / (total_k, Hk, D) tensors, lse (H, total_q).
  // The L2 / D vectors stay padded per (b, h) to Sq_pad rows.
  const int* cu_q;
  const int* cu_k;
  int total_q, total_k;
  // Dropout (DROP instances): the forward's keep flags; dV takes P o Z and
  // dS = P o (Z o dP - D), Z the kept entries' 1 / (1 - p) (0 where dropped).
  Dropout drop;
  int wl, wr;
  float scale;
  float scale_log2;
  unsigned int* status;
  uint64_t wait_ns;     // bounded-wait limit
  unsigned int inject;  // FA_INJECT_* (diagnostics only)
};

enum : uint32_t {
  SITE_KV_EMPTY = 0x31,
  SITE_KV_KV = 0x32,
  SITE_KV_QFULL = 0x33,
  SITE_KV_DOFULL = 0x34,
  SITE_KV_PD = 0x35,
  SITE_KV_SFREE = 0x36,
  SITE_KV_S = 0x37,
  SITE_KV_DP = 0x38,
  SITE_KV_ACC = 0x39,
  SITE_KV_DOEMPTY = 0x3A,
  SITE_KV_ALIGN = 0x3B,
  SITE_KV_FAC = 0x3C,
  SITE_KV_DS = 0x3D,
  SITE_KV_DQ = 0x3E,
  SITE_DQ_EMPTY = 0x41,
  SITE_DQ_Q = 0x42,
  SITE_DQ_K = 0x43,
  SITE_DQ_V = 0x44,
  SITE_DQ_DS = 0x45,
  SITE_DQ_S = 0x46,
  SITE_DQ_DP = 0x47,
  SITE_DQ_ACC = 0x48,
  SITE_DQ_ALIGN = 0x49,
  SITE_DQ_FAC = 0x4A,
};

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_load_w(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Timeout-only wait used while draining after an abort.
__device__ __forceinline__ void drain_wait_b(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// One sequence's lengths, first rows and TMA batch coordinate.
struct SeqInfo {
  int Sq, Sk, q_off, k_off, tb;
};
__device__ __forceinline__ SeqInfo seq_info(const BwdParams& p, int b) {
  if (!p.cu_q) return SeqInfo{p.Sq, p.Sk, 0, 0, b};
  const int q0 = p.cu_q[b], k0 = p.cu_k[b];
  return SeqInfo{p.cu_q[b + 1] - q0, p.cu_k[b + 1] - k0, q0, k0, 0};
}

// Does query tile qt meet key tile kt (does the bounding interval of its rows'
// live keys intersect the key tile)?
__device__ __forceinline__ bool qtile_meets(int qt, int kt, const BwdParams& p, int Sq, int Sk) {
  const int r0 = qt * 128;
  const int r1 = min(Sq, r0 + 128) - 1;
  const int lo = live_range(r0, Sq, Sk, p.wl, p.wr).lo;
  const int hi = live_range(r1, Sq, Sk, p.wl, p.wr).hi;
  if (hi < lo) return false;
  return !(hi < kt * 128 || lo > kt * 128 + 127);
}

// dS pair = P * (dP - D) with packed ops.
__device__ __forceinline__ void ds_pair(float p0, float p1, float dp0, float dp1, float d0, float d1, float& s0,
                                        float& s1) {
  f2_unpack(f2_mul(f2_pack(p0, p1), f2_sub(f2_pack(dp0, dp1), f2_pack(d0, d1))), s0, s1);
}

__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 u) {
  return make_uint4(bf16x2_to_f16x2(u.x), bf16x2_to_f16x2(u.y), bf16x2_to_f16x2(u.z), bf16x2_to_f16x2(u.w));
}

// ============================================================================ operand range
// The products run on fp16 copies of the bf16 inputs. fp16 has bf16's
// precision and more, but a far smaller range: normal from 2^-14 to 65504.
// Gradients with respect to the output are often 1e-5 .. 1e-8, where fp16
// loses most of its bits, and large inputs overflow. So each (sequence,
// key/value head) group of q, k, v and dout gets a power-of-two factor 2^e,
// copied as x * 2^e, which is exact wherever the product stays in fp16's
// normal range. The factors come back out exactly:
//   S'  = (Q 2^eq)(K 2^ek)^T = 2^(eq+ek) S       -> scale folded as 2^-(eq+ek)
//   dP' = (dO 2^edo)(V 2^ev)^T = 2^(edo+ev) dP    -> D kept as 2^(edo+ev) D
//   dS' = P o (dP' - D') = 2^(edo+ev) dS
//   dV' = P^T (dO 2^edo)                          -> times 2^-edo
//   dK' = dS'^T (Q 2^eq), dQ' = dS' (K 2^ek)      -> times scale 2^-(edo+ev+eq|ek)
// e puts the group's largest magnitude in [4, 8): then |dP'| <= |dO'_i| |V'_j|
// <= 64 D and |dS'| <= 128 D, inside fp16's range for D <= 128. A group
// already in [1, 8) keeps e = 0, so inputs of natural size are copied as they
// are. A group of zeros, or holding inf or NaN, keeps e = 0 too.
struct GroupExp {
  int q, k, v, dO;
};
// e for a group whose largest magnitude has bf16 bits `a` (sign cleared)
__device__ __forceinline__ int range_exp(uint32_t a) {
  if (a == 0 || a >= 0x7F80u) return 0;
  const int ef = int(a >> 7);  // biased exponent; 0 for subnormals (a * 2^-133)
  const int fl = ef > 0 ? ef - 127 : (31 - __clz(int(a & 0x7Fu))) - 133;  // floor(log2 |x|max)
  if (fl >= 0 && fl <= 2) return 0;
  return max(-120, min(120, 2 - fl));
}
__device__ __forceinline__ GroupExp group_exps(const uint32_t* amax, int b, int hk, int Hk) {
  const uint4 a = *reinterpret_cast<const uint4*>(amax + (size_t(b) * Hk + hk) * 4);
  return GroupExp{range_exp(a.x), range_exp(a.y), range_exp(a.z), range_exp(a.w)};
}
// 2^e as a float, |e| <= 126 (exact)
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float(uint32_t(127 + e) << 23); }
// scale * 2^-E as two factors m1 * m2, each exact; m2 = 1 unless |E| > 100, so
// x * m1 * m2 rounds once whenever the result can be represented at all.
__device__ __forceinline__ void unscale_factors(float scale, int E, float& m1, float& m2) {
  const int e1 = max(-100, min(100, E));
  m1 = scale * pow2f(-e1);
  m2 = pow2f(-max(-126, min(126, E - e1)));
}
// bf16 pair times m -> fp16 pair (exact while |x m| stays in fp16's normal range)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_mul(uint32_t v, float m) {
  return pack_f16x2(__uint_as_float(v << 16) * m, __uint_as_float(v & 0xFFFF0000u) * m);
}
__device__ __forceinline__ uint4 bf16x8_to_f16x8_mul(uint4 u, float m) {
  return make_uint4(bf16x2_to_f16x2_mul(u.x, m), bf16x2_to_f16x2_mul(u.y, m), bf16x2_to_f16x2_mul(u.z, m),
                    bf16x2_to_f16x2_mul(u.w, m));
}
// running max of the magnitudes of eight bf16 values, as two 16-bit halves
__device__ __forceinline__ uint32_t absmax8(uint32_t m, uint4 u) {
  m = __vmaxu2(m, u.x & 0x7FFF7FFFu);
  m = __vmaxu2(m, u.y & 0x7FFF7FFFu);
  m = __vmaxu2(m, u.z & 0x7FFF7FFFu);
  return __vmaxu2(m, u.w & 0x7FFF7FFFu);
}
// fp32 sum over eight element pairs of (a * ma) * (o * mo), in a fixed order
__device__ __forceinline__ float dot8_mul(uint4 a, uint4 o, float ma, float mo, float acc) {
  const uint32_t x[4] = {a.x, a.y, a.z, a.w};
  const uint32_t y[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    acc = fmaf(__uint_as_float(x[t] << 16) * ma, __uint_as_float(y[t] << 16) * mo, acc);
    acc = fmaf(__uint_as_float(x[t] & 0xFFFF0000u) * ma, __uint_as_float(y[t] & 0xFFFF0000u) * mo, acc);
  }
  return acc;
}

// Tokens per chunk of the rescale pass.
constexpr int CHUNK_TOK = 64;
// Replicas of each group's maxima in the pre-pass (block x writes replica x % AMAX_REPS).
constexpr int AMAX_REPS = 32;

// The query rows of one group in one chunk: items (token, head of the group,
// 16-byte chunk) with the chunk fastest, so a row's D/8 chunks sit on
// consecutive lanes of one warp. fn(live, token, g, element offset) runs on
// every lane, live or past the end; the loop is warp-uniform, so fn may shuffle.
template <int D, typename F>
__device__ __forceinline__ void for_q_items(const BwdParams& p, const SeqInfo& si, int b, int hk, int t0, F fn) {
  constexpr int CPR = D / 8;
  const long long per_tok = (long long)p.group * CPR;
  const int n_tok = max(0, min(CHUNK_TOK, si.Sq - t0));
  const long long items = n_tok * per_tok;
  const int lane = int(threadIdx.x & 31);
  for (long long base = (long long)threadIdx.x - lane; base < items; base += blockDim.x) {
    const long long it = base + lane;
    const int tl = int(it / per_tok);
    const long long rem = it - tl * per_tok;
    const size_t tok = p.cu_q ? size_t(si.q_off) + t0 + tl : size_t(b) * p.Sq + t0 + tl;
    fn(it < items, t0 + tl, int(rem / CPR), (tok * p.H + size_t(hk) * p.group) * D + size_t(rem) * 8);
  }
}
// The key rows of one key/value head in one chunk: items (token, chunk).
template <int D, typename F>
__device__ __forceinline__ void for_k_items(const BwdParams& p, const SeqInfo& si, int b, int hk, int t0, F fn) {
  constexpr int CPR = D / 8;
  const int n_tok = max(0, min(CHUNK_TOK, si.Sk - t0));
  const long long items = (long long)n_tok * CPR;
  for (long long it = threadIdx.x; it < items; it += blockDim.x) {
    const int tl = int(it / CPR);
    const size_t tok = p.cu_q ? size_t(si.k_off) + t0 + tl : size_t(b) * p.Sk + t0 + tl;
    fn((tok * p.Hk + hk) * D + size_t(it - (long long)tl * CPR) * 8);
  }
}

// Sequence holding packed token `tok` (last b with cu[b] <= tok), searched
// from b0, a sequence at or before it.
__device__ __forceinline__ int seq_of(const int* cu, int B, long long tok, int b0) {
  int lo = b0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= tok) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Largest magnitude over a row's R lanes (pairs of 16-bit magnitudes in), as
// one 16-bit magnitude; every lane of the warp must call it.
template <int R>
__device__ __forceinline__ uint32_t row_absmax(uint32_t m) {
#pragma unroll
  for (int off = R / 2; off > 0; off >>= 1) m = __vmaxu2(m, __shfl_xor_sync(0xffffffffu, m, off));
  return max(m & 0xFFFFu, m >> 16);
}
// Pre-pass, one 16-byte chunk (8 elements) of one row per item:
//   query rows: D_i = rowsum(dO_i o O_i), L2_i = L_i*log2(e) (+inf where L_i = -inf),
//               fp16 copies of Q_i and dO_i;
//   key rows:   fp16 copies of K_j and V_j;
//   padding:    D = 0 and L2 = +inf on the vector rows of each (b, h) past its
//               sequence, up to the whole 128-row tiles of Sq_pad;
//   range:      each row's largest |q|, |dO| (|k|, |v|) into one replica of its
//               group's maxima (amax_rep, zeroed before), through a running
//               maximum per thread that is sent when the thread changes group.
// The three item ranges start on multiples of 32, so each warp works inside one
// of them and the D/8 lanes of a row are consecutive lanes of one warp. The
// grid strides over the items, so the blocks sweep memory together. The copies
// are taken with e = 0; fa_bwd_rescale_kernel redoes those of groups that need
// a range factor.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const BwdParams p) {
  constexpr int CPR = D / 8;
  const long long rows_q = p.cu_q ? (long long)p.total_q : (long long)p.B * p.Sq;  // query tokens
  const long long rows_k = p.cu_q ? (long long)p.total_k : (long long)p.B * p.Sk;
  const long long n_q = rows_q * p.H * CPR;
  const long long k0 = (n_q + 31) & ~31LL;
  const long long n_k = rows_k * p.Hk * CPR;
  const long long p0 = (k0 + n_k + 31) & ~31LL;
  const long long n_pad = (long long)p.B * p.H * p.Sq_pad;
  const long long total = p0 + n_pad;
  const int lane = int(threadIdx.x & 31);
  const long long stride = (long long)gridDim.x * blockDim.x;
  // A row-leader thread's running maxima (m0, m1) of group cur (index * 2 +
  // side: 0 query rows (q, dO), 1 key rows (k, v)), kept in shared memory; they
  // go to the group's replica only when the thread moves to another group. With
  // long sequences the grid's stride keeps a thread on one group for many rows.
  __shared__ long long run_gid[256];
  __shared__ uint32_t run_max[256][2];
  run_gid[threadIdx.x] = -1;
  auto flush = [&]() {
    const long long cur = run_gid[threadIdx.x];
    if (cur < 0) return;
    uint32_t* g = p.amax_rep + ((size_t)(cur >> 1) * AMAX_REPS + blockIdx.x % AMAX_REPS) * 4;
    const bool key = cur & 1;
    if (run_max[threadIdx.x][0]) atomicMax(g + (key ? 1 : 0), run_max[threadIdx.x][0]);
    if (run_max[threadIdx.x][1]) atomicMax(g + (key ? 2 : 3), run_max[threadIdx.x][1]);
  };
  auto track = [&](long long gid, uint32_t m0, uint32_t m1) {
    if (run_gid[threadIdx.x] != gid) {
      flush();
      run_gid[threadIdx.x] = gid;
      run_max[threadIdx.x][0] = m0;
      run_max[threadIdx.x][1] = m1;
    } else {
      run_max[threadIdx.x][0] = max(run_max[threadIdx.x][0], m0);
      run_max[threadIdx.x][1] = max(run_max[threadIdx.x][1], m1);
    }
  };
  for (long long wb = ((long long)blockIdx.x * blockDim.x + threadIdx.x) - lane; wb < total; wb += stride) {
    const long long i = wb + lane;
    if (wb < k0) {
      const bool live = i < n_q;
      float acc = 0.0f;
      uint32_t mq = 0, mdo = 0;
      if (live) {
        const long long e = i * 8;  // = row * D + chunk * 8
        const uint4 qv = *reinterpret_cast<const uint4*>(p.q + e);
        const uint4 dov = *reinterpret_cast<const uint4*>(p.dout + e);
        const uint4 ov = *reinterpret_cast<const uint4*>(p.out + e);
        *reinterpret_cast<uint4*>(p.q16 + e) = bf16x8_to_f16x8_mul(qv, 1.0f);
        *reinterpret_cast<uint4*>(p.do16 + e) = bf16x8_to_f16x8_mul(dov, 1.0f);
        mq = absmax8(0, qv);
        mdo = absmax8(0, dov);
        acc = dot8_mul(dov, ov, 1.0f, 1.0f, 0.0f);
      }
#pragma unroll
      for (int off = CPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      mq = row_absmax<CPR>(mq);
      mdo = row_absmax<CPR>(mdo);
      if (live && (i % CPR) == 0) {
        const long long row = i / CPR;  // token * H + h
        const int h = int(row % p.H);
        const long long tok = row / p.H;
        int b, s;
        size_t li;
        if (p.cu_q) {  // the sequence holding this token: last b with cu_q[b] <= tok
          b = seq_of(p.cu_q, p.B, tok, 0);
          s = int(tok - p.cu_q[b]);
          li = size_t(h) * p.total_q + size_t(tok);
        } else {
          b = int(tok / p.Sq);
          s = int(tok % p.Sq);
          li = (size_t(b) * p.H + h) * p.Sq + s;
        }
        const size_t vi = (size_t(b) * p.H + h) * p.Sq_pad + s;
        p.dvec[vi] = acc;
        const float L = p.lse[li];
        p.nl2[vi] = (L == -INFINITY) ? -INFINITY : -(L * 1.4426950408889634f);
        track(((long long)b * p.Hk + h / p.group) * 2, mq, mdo);
      }
    } else if (wb < p0) {
      const long long t = i - k0;
      const bool live = t < n_k;
      uint32_t mk = 0, mv = 0;
      if (live) {
        const long long e = t * 8;
        const uint4 kv = *reinterpret_cast<const uint4*>(p.k + e);
        const uint4 vv = *reinterpret_cast<const uint4*>(p.v + e);
        *reinterpret_cast<uint4*>(p.k16 + e) = bf16x8_to_f16x8_mul(kv, 1.0f);
        *reinterpret_cast<uint4*>(p.v16 + e) = bf16x8_to_f16x8_mul(vv, 1.0f);
        mk = absmax8(0, kv);
        mv = absmax8(0, vv);
      }
      mk = row_absmax<CPR>(mk);
      mv = row_absmax<CPR>(mv);
      if (live && (t % CPR) == 0) {
        const long long row = t / CPR;  // token * Hk + hk
        const long long tok = row / p.Hk;
        const int b = p.cu_q ? seq_of(p.cu_k, p.B, tok, 0) : int(tok / p.Sk);
        track(((long long)b * p.Hk + (row - tok * p.Hk)) * 2 + 1, mk, mv);
      }
    } else {
      const long long t = i - p0;
      if (t < n_pad) {
        const int bh = int(t / p.Sq_pad), s = int(t % p.Sq_pad);
        const int b = bh / p.H;
        const int sq = p.cu_q ? p.cu_q[b + 1] - p.cu_q[b] : p.Sq;
        if (s >= sq) {
          p.dvec[t] = 0.0f;
          p.nl2[t] = -INFINITY;
        }
      }
    }
  }
  flush();
}

// Folds each group's replicas into its maxima (amax, block x = 0 writes them)
// and redoes the fp16 copies (and D) of the groups whose range factor is not
// 1. Block (x, hk, b) takes the 64-token chunks x, x + gridDim.x, ... of group
// (b, hk); a group that keeps e = 0 everywhere costs each of its blocks one
// read of its replicas.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_rescale_kernel(const BwdParams p) {
  constexpr int CPR = D / 8;
  const int lane = int(threadIdx.x & 31);
  const int hk = blockIdx.y, b = blockIdx.z;
  GroupExp ge;
  {
    // warp 0: lane r holds replica r; every warp computes the same maxima
    static_assert(AMAX_REPS == 32, "one replica per lane");
    const uint4 r = *reinterpret_cast<const uint4*>(p.amax_rep + (((size_t)b * p.Hk + hk) * AMAX_REPS + lane) * 4);
    uint32_t m[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m[t] = max(m[t], __shfl_xor_sync(0xffffffffu, m[t], off));
    if (blockIdx.x == 0 && threadIdx.x == 0)
      *reinterpret_cast<uint4*>(p.amax + ((size_t)b * p.Hk + hk) * 4) = make_uint4(m[0], m[1], m[2], m[3]);
    ge = GroupExp{range_exp(m[0]), range_exp(m[1]), range_exp(m[2]), range_exp(m[3])};
  }
  if ((ge.q | ge.k | ge.v | ge.dO) == 0) return;
  const SeqInfo si = seq_info(p, b);
  const float mq = pow2f(ge.q), mk = pow2f(ge.k), mv = pow2f(ge.v), mdo = pow2f(ge.dO);
  const bool redo_d = (ge.dO | ge.v) != 0;
  for (int chunk = blockIdx.x; chunk < p.n_chunks; chunk += gridDim.x) {
    const int t0 = chunk * CHUNK_TOK;
    if (ge.q | ge.dO | ge.v) {
      for_q_items<D>(p, si, b, hk, t0, [&](bool live, int s, int g, size_t e) {
        float acc = 0.0f;
        if (live) {
          if (ge.q)
            *reinterpret_cast<uint4*>(p.q16 + e) = bf16x8_to_f16x8_mul(*reinterpret_cast<const uint4*>(p.q + e), mq);
          if (redo_d) {
            const uint4 dov = *reinterpret_cast<const uint4*>(p.dout + e);
            if (ge.dO) *reinterpret_cast<uint4*>(p.do16 + e) = bf16x8_to_f16x8_mul(dov, mdo);
            // D' = rowsum((dO 2^edo) o (O 2^ev)): each factor scaled before the product
            acc = dot8_mul(dov, *reinterpret_cast<const uint4*>(p.out + e), mdo, mv, 0.0f);
          }
        }
        if (redo_d) {
#pragma unroll
          for (int off = CPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
          if (live && (lane % CPR) == 0) p.dvec[(size_t(b) * p.H + hk * p.group + g) * p.Sq_pad + s] = acc;
        }
      });
    }
    if (ge.k | ge.v) {
      for_k_items<D>(p, si, b, hk, t0, [&](size_t e) {
        if (ge.k)
          *reinterpret_cast<uint4*>(p.k16 + e) = bf16x8_to_f16x8_mul(*reinterpret_cast<const uint4*>(p.k + e), mk);
        if (ge.v)
          *reinterpret_cast<uint4*>(p.v16 + e) = bf16x8_to_f16x8_mul(*reinterpret_cast<const uint4*>(p.v + e), mv);
      });
    }
  }
}

// ============================================================================ dK / dV
// FDQ: the dK/dV kernel also forms each query tile's share of dQ (dS K over
// this CTA's 128 keys, M = queries) and adds it into an fp32 accumulator with a
// TMA reduction (page "FlashAttention：快速且内存高效的准确注意力机制", section
// "并行性 / 反向传播": dQ is summed across the key blocks). D = 64 only: TMEM then
// has room for the dQ tile beside S^T, one dP^T buffer, dV and dK.
template <int D, bool FDQ = false>
struct KvCfg {
  static_assert(!FDQ || D == 64, "the fused dQ fits TMEM at D = 64 only");
  static constexpr int PANELS = D / 64;
  static constexpr int PANEL_BYTES = 128 * 128;
  static constexpr int TILE_BYTES = PANELS * PANEL_BYTES;
  // Q of the next tile is read early (S^T of tile ii+1 is issued while tile ii
  // is still being processed), so Q gets a third stage; dO is read last. At
  // D = 64, dP^T of tile ii+1 also runs early (two dP^T buffers), and the
  // smaller tiles leave room for four stages of each.
  static constexpr int NQ = D == 64 ? 4 : 3;                    // Q stages
  static constexpr int NDO = D == 64 ? (FDQ ? 3 : 4) : 2;       // dO (+ L2, D) stages
  static constexpr int NDP = (D == 64 && !FDQ) ? 2 : 1;         // dP^T buffers in TMEM
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = TILE_BYTES;
  static constexpr int Q_OFF = 2 * TILE_BYTES;
  static constexpr int DO_OFF = Q_OFF + NQ * TILE_BYTES;
  static constexpr int VEC_OFF = DO_OFF + NDO * TILE_BYTES;  // per dO stage: L2[128], D[128]
  // Compute warpgroups; each owns COLS query columns. Without FDQ, two halve
  // the per-tile bookkeeping (waits, fences, arrives, addresses) per element
  // against four: 20% fewer instructions, 1% (D = 64) to 4% (D = 128) faster at
  // S = 4096. FDQ lengthens each tile's compute chain (dS to shared memory, the
  // dQ reduction), and four groups hide more of its latency.
  static constexpr int NCW = FDQ ? 4 : 2;
  static constexpr int COLS = 128 / NCW;
  static constexpr int NCT = 128 * NCW;  // compute threads
  // FDQ: dS of the tile as the dQ MMA's A operand (M = 128 queries in two
  // 64-query panels of 128 key rows, MN-major, 128-byte swizzled), and per
  // compute warp a 32-row x DQC-column fp32 staging box for its reduction
  // (group w reduces dQ columns w*DQC .. w*DQC + DQC - 1).
  static constexpr int DQC = D / NCW;
  static constexpr int DS_OFF = VEC_OFF + NDO * 1024;
  static constexpr int DS_BYTES = FDQ ? 2 * PANEL_BYTES : 0;
  static constexpr int STG_OFF = DS_OFF + DS_BYTES;
  static constexpr int STG_BYTES = FDQ ? NCT * DQC * 4 : 0;
  static constexpr int BAR_OFF = STG_OFF + STG_BYTES;
  static constexpr int SMEM_BYTES = BAR_OFF + 320;
  static constexpr int THREADS = 128 + NCT;
  static constexpr int DO_TX = TILE_BYTES + 1024;
  // TMEM: S^T [0,128) fp32; dP^T of tile ii in buffer ii % NDP at
  // [128 + 128 b, 256 + 128 b) fp32, over which, once consumed, the 16-query
  // chunk kk of P^T (fp16 pairs) sits at columns 16kk+0..7 and that of dS^T at
  // 16kk+8..15, so every compute group writes only inside the dP^T columns it
  // has read itself; dV and dK accumulators after the buffers. With two
  // buffers, S^T and dP^T of tile ii+1 run on the tensor pipe while the
  // compute groups form P^T and dS^T of tile ii.
  // FDQ: the tile's dQ share (lanes = query rows) after dK.
  static constexpr uint32_t T_S = 0, T_DP = 128, T_DV = 128 + 128 * NDP, T_DK = T_DV + D, T_DQ = T_DK + D;
  static_assert(T_DK + D + (FDQ ? D : 0) <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(!FDQ || DQC == 16 || DQC == 32, "staging rows of 64 or 128 bytes (the map's swizzle span)");
};

struct KvBars {
  uint64_t kv_full;
  uint64_t q_full[4], q_empty[4];
  uint64_t do_full[4], do_empty[4];
  uint64_t s_full, s_free, acc_done, drain;
  uint64_t dp_full[2], pd_ready[2];  // per dP^T buffer
  uint64_t fac_ready;                 // fac[] written (warp 2)
  uint64_t ds_ready, dq_full;         // FDQ: dS in shared memory; the tile's dQ share done
  float fac[6];                       // scale_log2 for S^T, dV factor, dK factors m1, m2, dQ factors m1, m2
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(KvBars) <= 320, "barrier block");

// FDQ: tm_dqa maps the fp32 dQ accumulator (B, Sq, H, D) in boxes of DQC columns
// (one compute group's share of D) x 32 rows, 64-byte swizzled; otherwise unused.
template <int D, bool DROP, bool FDQ>
__global__ void __launch_bounds__(KvCfg<D, FDQ>::THREADS, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dqa, const BwdParams p) {
  using C = KvCfg<D, FDQ>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // the swizzled layouts need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(p.status, FA_DEV_TIMEOUT | SITE_KV_ALIGN);
    return;
  }
  KvBars* bars = reinterpret_cast<KvBars*>(smem + C::BAR_OFF);
  const int warp = int(warp_id());
  const int lane = int(lane_id());
  const int kt = blockIdx.x;
  const int hk = blockIdx.y;  // key/value head; its query heads are hk*group .. hk*group + group - 1
  const int b = blockIdx.z;
  const int j0 = kt * 128;
  const SeqInfo sq_ = seq_info(p, b);
  const int Sq = sq_.Sq, Sk = sq_.Sk;
  if (j0 >= Sk) return;  // shorter than the longest key sequence: no keys here
  const int n_qt = (Sq + 127) / 128;

  // Live query tiles of this key tile: a contiguous range, the same for every
  // query head. Iteration ii covers query head hk*group + ii / n_qtl and query
  // tile qt_first + ii % n_qtl (the loops step both), so the group's dK, dV sums
  // stay in this CTA.
  int qt_first = n_qt, qt_last = -1;
  for (int qt = 0; qt < n_qt; ++qt) {
    if (qtile_meets(qt, kt, p, Sq, Sk)) {
      qt_first = min(qt_first, qt);
      qt_last = qt;
    }
  }
  const int n_qtl = qt_last >= qt_first ? qt_last - qt_first + 1 : 0;
  const int n_iter = n_qtl * p.group;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < C::NQ; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
    }
    for (int s = 0; s < C::NDO; ++s) {
      mbar_init(&bars->do_full[s], 1);
      mbar_init(&bars->do_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, C::NCT / 32);  // one arrive per compute warp
    for (int s = 0; s < C::NDP; ++s) {
      mbar_init(&bars->dp_full[s], 1);
      mbar_init(&bars->pd_ready[s], C::NCT / 32);
    }
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->fac_ready, 1);
    mbar_init(&bars->ds_ready, C::NCT / 32);  // one arrive per compute warp
    mbar_init(&bars->dq_full, 1);
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
    if (n_iter > 0) {
      tma_prefetch_desc_w(&tm_q);
      tma_prefetch_desc_w(&tm_k);
      tma_prefetch_desc_w(&tm_v);
      tma_prefetch_desc_w(&tm_do);
      mbar_arrive_expect_tx_w(&bars->kv_full, 2 * C::TILE_BYTES);
      for (int pn = 0; pn < C::PANELS; ++pn) {
        tma_load_4d_w(smem + C::K_OFF + pn * C::PANEL_BYTES, &tm_k, &bars->kv_full, pn * 64, hk, sq_.k_off + j0,
                    sq_.tb);
        tma_load_4d_w(smem + C::V_OFF + pn * C::PANEL_BYTES, &tm_v, &bars->kv_full, pn * 64, hk, sq_.k_off + j0,
                    sq_.tb);
      }
      int q_issued = 0, do_issued = 0;
      // query head and tile of iteration ii, stepped instead of divided out
      int hq = hk * p.group, qt = qt_first;
      for (int ii = 0; ii < n_iter; ++ii, qt = (qt == qt_last) ? (++hq, qt_first) : qt + 1) {
        const int s = ii % C::NQ;
        const int i0 = qt * 128;
        const size_t vec_base = (size_t(b) * p.H + hq) * p.Sq_pad;
        if (!fa_wait_warp(&bars->q_empty[s], (uint32_t(ii / C::NQ) & 1u) ^ 1u, watch, SITE_KV_EMPTY)) break;
        mbar_arrive_expect_tx_w(&bars->q_full[s], C::TILE_BYTES);
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d_w(smem + C::Q_OFF + s * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_q, &bars->q_full[s], pn * 64,
                      hq, sq_.q_off + i0, sq_.tb);
        q_issued = ii + 1;
        const int d = ii % C::NDO;
        if (!fa_wait_warp(&bars->do_empty[d], (uint32_t(ii / C::NDO) & 1u) ^ 1u, watch, SITE_KV_DOEMPTY)) break;
        mbar_arrive_expect_tx_w(&bars->do_full[d], C::DO_TX);
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d_w(smem + C::DO_OFF + d * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_do, &bars->do_full[d],
                      pn * 64, hq, sq_.q_off + i0, sq_.tb);
        bulk_load_w(smem + C::VEC_OFF + d * 1024, p.nl2 + vec_base + i0, 512, &bars->do_full[d]);
        bulk_load_w(smem + C::VEC_OFF + d * 1024 + 512, p.dvec + vec_base + i0, 512, &bars->do_full[d]);
        do_issued = ii + 1;
      }
      // every copy must land before the CTA may exit
      drain_wait_b(&bars->kv_full, 0, p.wait_ns);
      for (int ii = (q_issued > C::NQ ? q_issued - C::NQ : 0); ii < q_issued; ++ii)
        drain_wait_b(&bars->q_full[ii % C::NQ], uint32_t(ii / C::NQ) & 1u, p.wait_ns);
      for (int ii = (do_issued > C::NDO ? do_issued - C::NDO : 0); ii < do_issued; ++ii)
        drain_wait_b(&bars->do_full[ii % C::NDO], uint32_t(ii / C::NDO) & 1u, p.wait_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Descriptors are built once; each k-step and stage is a constant added to
    // the start-address field, so issuing keeps pace with the tensor pipe.
    // The whole warp runs the loop; one elected lane issues each MMA and commit.
    if (n_iter > 0) {
      constexpr uint32_t ID_SS = idesc_f16_f32(128, 128, 0, 0);  // S^T, dP^T: both operands K-major
      constexpr uint32_t ID_TN = idesc_f16_f32(128, D, 0, 1);    // dV, dK: A from TMEM, B (dO / Q) MN-major
      const uint64_t k_desc = sdesc_sw128(smem_u32(smem + C::K_OFF), 16, 1024);
      const uint64_t v_desc = sdesc_sw128(smem_u32(smem + C::V_OFF), 16, 1024);
      const uint64_t q_kdesc = sdesc_sw128(smem_u32(smem + C::Q_OFF), 16, 1024);     // Q as K-major (S^T)
      const uint64_t do_kdesc = sdesc_sw128(smem_u32(smem + C::DO_OFF), 16, 1024);   // dO as K-major (dP^T)
      const uint64_t q_mdesc = sdesc_sw128(smem_u32(smem + C::Q_OFF), C::PANEL_BYTES, 1024);    // MN-major (dK)
      const uint64_t do_mdesc = sdesc_sw128(smem_u32(smem + C::DO_OFF), C::PANEL_BYTES, 1024);  // MN-major (dV)
      // FDQ: dQ share = dS K, A = dS (queries x keys) and B = K (keys x D), both MN-major
      constexpr uint32_t ID_DQ = idesc_f16_f32(128, D, 1, 1);
      const uint64_t ds_desc = sdesc_sw128(smem_u32(smem + C::DS_OFF), C::PANEL_BYTES, 1024);
      const uint64_t k_mdesc = sdesc_sw128(smem_u32(smem + C::K_OFF), C::PANEL_BYTES, 1024);
      const uint32_t t_s = tmem + C::T_S, t_dp = tmem + C::T_DP, t_dv = tmem + C::T_DV, t_dk = tmem + C::T_DK;
      const uint32_t t_dq = tmem + C::T_DQ;
      // dP^T(ii) = V dO^T into buffer ii % NDP
      auto issue_dp = [&](int ii) {
        if (!fa_wait_warp(&bars->do_full[ii % C::NDO], uint32_t(ii / C::NDO) & 1u, watch, SITE_KV_DOFULL))
          return false;
        tc_fence_after();
        const uint64_t dod = sdesc_adv(do_kdesc, uint32_t(ii % C::NDO) * C::TILE_BYTES);
        const uint32_t dst = t_dp + uint32_t(ii % C::NDP) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::PANEL_BYTES + (kk % 4) * 32;
          mma_ss_w(dst, sdesc_adv(v_desc, off), sdesc_adv(dod, off), ID_SS, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(&bars->dp_full[ii % C::NDP]);
        return true;
      };
      bool ok = fa_wait_warp(&bars->kv_full, 0, watch, SITE_KV_KV) && fa_wait_warp(&bars->q_full[0], 0, watch, SITE_KV_QFULL);
      if (ok) {  // S^T(0) = K Q^T
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::PANEL_BYTES + (kk % 4) * 32;
          mma_ss_w(t_s, sdesc_adv(k_desc, off), sdesc_adv(q_kdesc, off), ID_SS, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(&bars->s_full);
      }
      ok = ok && issue_dp(0);
      for (int ii = 0; ii < n_iter && ok; ++ii) {
        const bool more = ii + 1 < n_iter;
        const uint32_t q_cur = uint32_t(ii % C::NQ) * C::TILE_BYTES;        // Q stage of tile ii
        const uint32_t q_nxt = uint32_t((ii + 1) % C::NQ) * C::TILE_BYTES;  // Q stage of tile ii + 1
        const uint32_t do_cur = uint32_t(ii % C::NDO) * C::TILE_BYTES;
        // S^T of the next tile as soon as every compute group holds this one in registers
        if (more) {
          if (!(ok = fa_wait_warp(&bars->s_free, uint32_t(ii) & 1u, watch, SITE_KV_SFREE))) break;
          if (!(ok = fa_wait_warp(&bars->q_full[(ii + 1) % C::NQ], uint32_t((ii + 1) / C::NQ) & 1u, watch,
                             SITE_KV_QFULL)))
            break;
          tc_fence_after();
          const uint64_t qd = sdesc_adv(q_kdesc, q_nxt);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * C::PANEL_BYTES + (kk % 4) * 32;
            mma_ss_w(t_s, sdesc_adv(k_desc, off), sdesc_adv(qd, off), ID_SS, kk > 0 ? 1u : 0u);
          }
          mma_commit_w(&bars->s_full);
          // with a second buffer, dP^T of the next tile too; it overwrites the
          // buffer of tile ii-1, whose dV, dK were issued before (read in order)
          if (C::NDP == 2 && !(ok = issue_dp(ii + 1))) break;
        }
        // dV += P^T dO and dK += dS^T Q, two independent chains; the 16-query chunk kk
        // of P^T sits at dP^T column 16kk of its buffer, that of dS^T at 16kk+8
        const int pb = ii % C::NDP;
        if (!(ok = fa_wait_warp(&bars->pd_ready[pb], uint32_t(ii / C::NDP) & 1u, watch, SITE_KV_PD))) break;
        tc_fence_after();
        {
          const uint64_t dod = sdesc_adv(do_mdesc, do_cur), qd = sdesc_adv(q_mdesc, q_cur);
          const uint32_t src = t_dp + uint32_t(pb) * 128;
          const uint32_t acc0 = ii > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            mma_ts_w(t_dv, src + kk * 16, sdesc_adv(dod, kk * 2048), ID_TN, kk > 0 ? 1u : acc0);
            mma_ts_w(t_dk, src + kk * 16 + 8, sdesc_adv(qd, kk * 2048), ID_TN, kk > 0 ? 1u : acc0);
          }
        }
        mma_commit_w(&bars->do_empty[ii % C::NDO]);
        mma_commit_w(&bars->q_empty[ii % C::NQ]);
        // with one buffer, dP^T of the next tile overwrites P^T and dS^T of this
        // one, read above (in order)
        if (C::NDP == 1 && more && !(ok = issue_dp(ii + 1))) break;
        if constexpr (FDQ) {
          // this tile's dQ share over the CTA's 128 keys, from scratch, once dS is in
          // shared memory; behind dP^T of the next tile, so that one reaches the
          // compute warps first. They read the share (dq_full) during the next
          // tile, before they arrive on its ds_ready, which the next share waits for.
          if (!(ok = fa_wait_warp(&bars->ds_ready, uint32_t(ii) & 1u, watch, SITE_KV_DS))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss_w(t_dq, sdesc_adv(ds_desc, kk * 2048), sdesc_adv(k_mdesc, kk * 2048), ID_DQ, kk > 0 ? 1u : 0u);
          mma_commit_w(&bars->dq_full);
        }
      }
      if (ok) {
        mma_commit_w(&bars->acc_done);
      } else {
        mma_commit_w(&bars->drain);
        drain_wait_b(&bars->drain, 0, p.wait_ns);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ range factors of the group
    if (lane == 0) {
      const GroupExp ge = group_exps(p.amax, b, hk, p.Hk);
      bars->fac[0] = p.scale_log2 * pow2f(-ge.q) * pow2f(-ge.k);
      bars->fac[1] = pow2f(-ge.dO);
      unscale_factors(p.scale, ge.dO + ge.v + ge.q, bars->fac[2], bars->fac[3]);
      unscale_factors(p.scale, ge.dO + ge.v + ge.k, bars->fac[4], bars->fac[5]);  // dQ' = 2^(edo+ev+ek) dQ / scale
      mbar_arrive(&bars->fac_ready);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ compute (thread = key row)
    const int w = (warp - 4) / 4;  // query-column group: columns [w*COLS, (w+1)*COLS)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int j = j0 + r;
    const uint32_t lane_addr = uint32_t(wq * 32) << 16;
    const int off = Sk - Sq;
    // live queries of key j: i in [qlo, qhi]
    auto qbounds = [&](int jj, int& lo, int& hi) {
      lo = (p.wr >= 0) ? jj - off - p.wr : 0;
      hi = (p.wl >= 0) ? jj - off + p.wl : Sq - 1;
      lo = max(lo, 0);
      hi = min(hi, Sq - 1);
      if (jj >= Sk) {
        lo = 1;
        hi = 0;
      }
    };
    int qlo, qhi;
    qbounds(j, qlo, qhi);
    int qlo_max, dummy, qhi_min;
    qbounds(min(Sk - 1, j0 + 127), qlo_max, dummy);
    qbounds(j0, dummy, qhi_min);
    const bool tile_keys_ok = j0 + 127 < Sk;
    const bool has_alibi = p.alibi != nullptr;
    // the group's range factors (warp 2): S^T arrives as 2^(eq+ek) S^T
    bool ok = fa_wait_warp(&bars->fac_ready, 0, watch, SITE_KV_FAC);
    const float sl = bars->fac[0];
    // FDQ: a tile's dQ share (TMEM lanes = query rows; group w takes DQC
    // columns from w * DQC), times the unscaling factors, into the warp's staging
    // box (its 32 rows at DQC * 4 bytes each, swizzled as the accumulator's
    // tensor map is: 16-byte chunk c of row l at c ^ (l & 7) for 128-byte rows,
    // c ^ ((l >> 1) & 3) for 64-byte rows), then one TMA reduction of the box into
    // the fp32 accumulator, issued by lane 0. Before the box is written again,
    // lane 0 waits until its last reduction has read it.
    constexpr int RB = C::DQC * 4;  // staging row bytes
    uint8_t* stg = smem + C::STG_OFF + (w * 4 + wq) * (32 * RB);
    const int sw = RB == 128 ? (lane & 7) : ((lane >> 1) & 3);
    auto reduce_dq = [&](int hq_t, int i0_t) {
      float a[C::DQC];
      tmem_ld_cols(tmem + lane_addr + C::T_DQ + uint32_t(w * C::DQC), a);
      if (lane == 0) bulk_wait_group_read0();
      __syncwarp();
      const float m1 = bars->fac[4], m2 = bars->fac[5];
#pragma unroll
      for (int c = 0; c < C::DQC / 4; ++c) {
        float4 v;
        if (m2 == 1.0f) {  // the usual case (|E| <= 100): x * m1 * m2 is x * m1
          v = make_float4(a[4 * c] * m1, a[4 * c + 1] * m1, a[4 * c + 2] * m1, a[4 * c + 3] * m1);
        } else {
          v = make_float4(a[4 * c] * m1 * m2, a[4 * c + 1] * m1 * m2, a[4 * c + 2] * m1 * m2, a[4 * c + 3] * m1 * m2);
        }
        *reinterpret_cast<float4*>(stg + lane * RB + ((c ^ sw) * 16)) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_reduce_add_4d(&tm_dqa, stg, w * C::DQC, hq_t, i0_t + wq * 32, b);
        bulk_commit_group();
      }
      __syncwarp();
    };
    int hq_prev = 0, i0_prev = 0;  // FDQ: the previous tile's query head and first row
    // query head and tile of iteration ii, stepped instead of divided out
    int hq = hk * p.group, qt = qt_first;
    for (int ii = 0; ii < n_iter && ok; ++ii, qt = (qt == qt_last) ? (++hq, qt_first) : qt + 1) {
      const int d = ii % C::NDO;
      const int i0 = qt * 128;
      const float slope_log2 = has_alibi ? p.alibi[b * p.alibi_bstride + hq] * 1.4426950408889634f : 0.0f;
      const int ib = i0 + w * C::COLS;  // first query of this group
      const float4* nl2v = reinterpret_cast<const float4*>(smem + C::VEC_OFF + d * 1024) + w * (C::COLS / 4);
      const float4* dvv = nl2v + 32;
      // the L2 / D vectors of this tile land with dO
      if (!(ok = fa_wait_warp(&bars->do_full[d], uint32_t(ii / C::NDO) & 1u, watch, SITE_KV_DOFULL))) break;
      if (!(ok = fa_wait_warp(&bars->s_full, uint32_t(ii) & 1u, watch, SITE_KV_S))) break;
      tc_fence_after();
      float pv[C::COLS];
      tmem_ld_cols(tmem + lane_addr + C::T_S + w * C::COLS, pv);
      tc_fence_before();
      mbar_arrive_warp(&bars->s_free);
      const bool need_mask = !(tile_keys_ok && i0 >= qlo_max && i0 + 127 <= qhi_min);
      const uint64_t sl2 = f2_pack(sl, sl);
      const int dd0 = ib + off - j;  // c(i) - j for the group's first query
      if (has_alibi && (dd0 >= 0 || dd0 + C::COLS - 1 <= 0)) {
        // ALiBi with this key's queries all on one side of the diagonal:
        // slope * |c(i) - j| = (+-slope) * (c(i) - j) runs on column pairs,
        // rounding as the scalar form below does (the distances are exact).
        const float ms = dd0 >= 0 ? slope_log2 : -slope_log2;
        const uint64_t ms2 = f2_pack(ms, ms), st2 = f2_pack(4.0f, 4.0f);
        uint64_t distA = f2_pack(float(dd0), float(dd0) + 1.0f);
        uint64_t distB = f2_pack(float(dd0) + 2.0f, float(dd0) + 3.0f);
#pragma unroll
        for (int c4 = 0; c4 < C::COLS / 4; ++c4) {
          const float4 l4 = nl2v[c4];
          const uint64_t bA = f2_sub(f2_pack(l4.x, l4.y), f2_mul(distA, ms2));
          const uint64_t bB = f2_sub(f2_pack(l4.z, l4.w), f2_mul(distB, ms2));
          distA = f2_add(distA, st2);
          distB = f2_add(distB, st2);
          float a0, a1, a2, a3;
          f2_unpack(f2_fma(f2_pack(pv[4 * c4], pv[4 * c4 + 1]), sl2, bA), a0, a1);
          f2_unpack(f2_fma(f2_pack(pv[4 * c4 + 2], pv[4 * c4 + 3]), sl2, bB), a2, a3);
          pv[4 * c4] = ex2_approx(a0);
          pv[4 * c4 + 1] = ex2_approx(a1);
          pv[4 * c4 + 2] = ex2_approx(a2);
          pv[4 * c4 + 3] = ex2_approx(a3);
        }
      } else if (has_alibi) {
#pragma unroll
        for (int c4 = 0; c4 < C::COLS / 4; ++c4) {
          const float4 l4 = nl2v[c4];
          const float dd = float(dd0 + 4 * c4);
          const float b0 = l4.x - slope_log2 * fabsf(dd);
          const float b1 = l4.y - slope_log2 * fabsf(dd + 1.0f);
          const float b2 = l4.z - slope_log2 * fabsf(dd + 2.0f);
          const float b3 = l4.w - slope_log2 * fabsf(dd + 3.0f);
          float a0, a1, a2, a3;
          f2_unpack(f2_fma(f2_pack(pv[4 * c4], pv[4 * c4 + 1]), sl2, f2_pack(b0, b1)), a0, a1);
          f2_unpack(f2_fma(f2_pack(pv[4 * c4 + 2], pv[4 * c4 + 3]), sl2, f2_pack(b2, b3)), a2, a3);
          pv[4 * c4] = ex2_approx(a0);
          pv[4 * c4 + 1] = ex2_approx(a1);
          pv[4 * c4 + 2] = ex2_approx(a2);
          pv[4 * c4 + 3] = ex2_approx(a3);
        }
      } else {
        // the stored bias pairs feed the paired FMA as they are
#pragma unroll
        for (int c4 = 0; c4 < C::COLS / 4; ++c4) {
          const float4 l4 = nl2v[c4];
          float a0, a1, a2, a3;
          f2_unpack(f2_fma(f2_pack(pv[4 * c4], pv[4 * c4 + 1]), sl2, f2_pack(l4.x, l4.y)), a0, a1);
          f2_unpack(f2_fma(f2_pack(pv[4 * c4 + 2], pv[4 * c4 + 3]), sl2, f2_pack(l4.z, l4.w)), a2, a3);
          pv[4 * c4] = ex2_approx(a0);
          pv[4 * c4 + 1] = ex2_approx(a1);
          pv[4 * c4 + 2] = ex2_approx(a2);
          pv[4 * c4 + 3] = ex2_approx(a3);
        }
      }
      if (need_mask) {
        const int lo = qlo - ib, hi = qhi - ib;
#pragma unroll
        for (int c = 0; c < C::COLS; ++c) pv[c] = (c >= lo && c <= hi) ? pv[c] : 0.0f;
      }
      const int pb = ii % C::NDP;
      if (!(ok = fa_wait_warp(&bars->dp_full[pb], uint32_t(ii / C::NDP) & 1u, watch, SITE_KV_DP))) break;
      tc_fence_after();
      // per 16-query chunk: load dP^T, form dS^T, then P^T and dS^T as fp16 pairs over
      // the chunk's consumed dP^T columns (see the TMEM map)
      uint32_t ds_all[FDQ ? C::COLS / 2 : 1];  // FDQ: the tile's dS, kept for shared memory
#pragma unroll
      for (int ch = 0; ch < C::COLS / 16; ++ch) {
        float dp[16];
        const uint32_t col = tmem + lane_addr + C::T_DP + uint32_t(pb) * 128 + w * C::COLS + 16 * ch;
        tmem_ld_cols(col, dp);
        uint32_t pp[8], ps[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = 16 * ch + 2 * e;
          const float4 d4 = dvv[c / 4];
          const float dv0 = (c % 4 == 0) ? d4.x : d4.z;
          const float dv1 = (c % 4 == 0) ? d4.y : d4.w;
          float s0, s1;
          if constexpr (DROP) {  // this key's flags for query rows ib + c and ib + c + 1
            const int bh = b * p.H + hq;
            const float z0 = (dropout_keep4(p.drop, bh, ib + c, j >> 2) >> (j & 3)) & 1u ? p.drop.keep_scale : 0.0f;
            const float z1 =
                (dropout_keep4(p.drop, bh, ib + c + 1, j >> 2) >> (j & 3)) & 1u ? p.drop.keep_scale : 0.0f;
            ds_pair(pv[c], pv[c + 1], dp[2 * e] * z0, dp[2 * e + 1] * z1, dv0, dv1, s0, s1);
            pp[e] = pack_f16x2(pv[c] * z0, pv[c + 1] * z1);
          } else {
            ds_pair(pv[c], pv[c + 1], dp[2 * e], dp[2 * e + 1], dv0, dv1, s0, s1);
            pp[e] = pack_f16x2(pv[c], pv[c + 1]);
          }
          ps[e] = pack_f16x2(s0, s1);
        }
        tmem_st_x8(col, pp);
        tmem_st_x8(col + 8, ps);
        if constexpr (FDQ) {
#pragma unroll
          for (int e = 0; e < 8; ++e) ds_all[8 * ch + e] = ps[e];
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(&bars->pd_ready[pb]);
      if constexpr (FDQ) {
        // The last tile's dQ share is complete (and has read the dS buffer): add it
        // into the accumulator, then this tile's dS as the dQ MMA's A operand: key
        // row r of the 64-query panel holding the group's queries, from 16-byte
        // chunk (w * COLS % 64) / 8.
        if (ii > 0) {
          if (!(ok = fa_wait_warp(&bars->dq_full, uint32_t(ii - 1) & 1u, watch, SITE_KV_DQ))) break;
          tc_fence_after();
          reduce_dq(hq_prev, i0_prev);
        }
        uint8_t* ds_row = smem + C::DS_OFF + (w * C::COLS / 64) * C::PANEL_BYTES + r * 128;
        const int ck0 = (w * C::COLS % 64) / 8;
#pragma unroll
        for (int ch = 0; ch < C::COLS / 16; ++ch) {
          const uint32_t* v = ds_all + 8 * ch;
          *reinterpret_cast<uint4*>(ds_row + (((ck0 + 2 * ch) ^ (r & 7)) * 16)) = make_uint4(v[0], v[1], v[2], v[3]);
          *reinterpret_cast<uint4*>(ds_row + (((ck0 + 2 * ch + 1) ^ (r & 7)) * 16)) =
              make_uint4(v[4], v[5], v[6], v[7]);
        }
        fence_proxy_async_smem();  // dS is read by the tensor core next
        tc_fence_before();         // and the share's TMEM columns are rewritten by the next share
        mbar_arrive_warp(&bars->ds_ready);
      }
      hq_prev = hq;
      i0_prev = i0;
    }
    // ------------------------------------------------------------ dK / dV epilogue
    // groups 0..NCW/2-1 write dV, the rest dK (times scale); each a D/(NCW/2)-column slice
    constexpr int SLICE = D / (C::NCW / 2);
    const bool is_dv = w < C::NCW / 2;
    const int col0 = (w % (C::NCW / 2)) * SLICE;
    // read again rather than kept live across the loop
    const SeqInfo e_sq = seq_info(p, b);
    const bool row_ok = j < e_sq.Sk;
    const size_t krow = p.cu_q ? size_t(e_sq.k_off) + j : size_t(b) * e_sq.Sk + j;
    __nv_bfloat16* dst = (is_dv ? p.dv : p.dk) + (krow * p.Hk + hk) * size_t(D) + col0;
    // dV' = 2^edo dV, dK' = 2^(edo+ev+eq) dK / scale
    const float mul = is_dv ? bars->fac[1] : bars->fac[2];
    const float mul2 = is_dv ? 1.0f : bars->fac[3];
    if (n_iter == 0) {
      if (row_ok)
        for (int e = 0; e < SLICE / 8; ++e) reinterpret_cast<uint4*>(dst)[e] = make_uint4(0, 0, 0, 0);
    } else if (ok && fa_wait_warp(&bars->acc_done, 0, watch, SITE_KV_ACC)) {
      tc_fence_after();
      if constexpr (FDQ) reduce_dq(hq_prev, i0_prev);  // the last tile's dQ share (acc_done follows it)
#pragma unroll 1
      for (int cc = 0; cc < SLICE / 32; ++cc) {
        float a[32];
        tmem_ld_x32f(tmem + lane_addr + (is_dv ? C::T_DV : C::T_DK) + col0 + cc * 32, a);
        if (row_ok) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(a[2 * e] * mul * mul2, a[2 * e + 1] * mul * mul2);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            reinterpret_cast<uint4*>(dst + cc * 32)[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
    }
    // every reduction this warp issued has landed before the CTA ends
    if (FDQ && lane == 0) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================================ dQ
template <int D>
struct DqCfg {
  static constexpr int PANELS = D / 64;
  static constexpr int PANEL_BYTES = 128 * 128;
  static constexpr int TILE_BYTES = PANELS * PANEL_BYTES;
  // K_j stays until dQ(j) has read it, V_j only until dP(j); separate rings let
  // V of a later tile load as soon as dP has freed a slot.
  static constexpr int NK = D == 64 ? 4 : 3;  // ring of K_j tiles
  static constexpr int NV = D == 64 ? 4 : 2;  // ring of V_j tiles
  static constexpr int Q_OFF = 0;
  static constexpr int DO_OFF = TILE_BYTES;
  static constexpr int K_OFF = 2 * TILE_BYTES;
  static constexpr int V_OFF = K_OFF + NK * TILE_BYTES;
  static constexpr int BAR_OFF = V_OFF + NV * TILE_BYTES;
  static constexpr int SMEM_BYTES = BAR_OFF + 256;
  // Compute warpgroups; each owns COLS key columns. Two at D = 128 (3.5% faster
  // than four at S = 4096); four at D = 64, where shorter per-warp chains hide
  // more of the per-tile latency (two were 1.3% slower).
  static constexpr int NCW = D == 64 ? 4 : 2;
  static constexpr int COLS = 128 / NCW;
  static constexpr int NCT = 128 * NCW;
  static constexpr int THREADS = 128 + NCT;
  // TMEM: S at [0,128); dP of tile j in buffer j % 2 at [128,256) or [256,384);
  // dQ at [384,384+D). Once dP is consumed, the 16-key chunk kk of dS (fp16
  // pairs) sits at its buffer's columns 16kk+0..7, inside the columns its compute
  // group has read itself. S is free as soon as every group holds it in
  // registers; with two dP buffers, S and dP of tile j+1 run on the tensor pipe
  // while the compute groups form dS of tile j.
  static constexpr int NDP = 2;
  static constexpr uint32_t T_S = 0, T_DP = 128, T_DQ = 128 + 128 * NDP;
  static_assert(T_DQ + D <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct DqBars {
  uint64_t q_full;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full, s_free, acc_done, drain;
  uint64_t dp_full[2], ds_ready[2];  // per dP buffer
  uint64_t fac_ready;                 // fac[] written (warp 2)
  float fac[4];                       // scale_log2 for S, dQ factors m1, m2
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(DqBars) <= 256, "barrier block");

template <int D, bool DROP>
__global__ void __launch_bounds__(DqCfg<D>::THREADS, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const BwdParams p) {
  using C = DqCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, FA_DEV_TIMEOUT | SITE_DQ_ALIGN);
    return;
  }
  DqBars* bars = reinterpret_cast<DqBars*>(smem + C::BAR_OFF);
  const int warp = int(warp_id());
  const int lane = int(lane_id());
  const int h = blockIdx.y;
  const int hkv = h / p.group;  // key/value head of this query head
  const int b = blockIdx.z;
  const SeqInfo sq_ = seq_info(p, b);
  const int Sq = sq_.Sq, Sk = sq_.Sk;
  const int n_qt = (Sq + 127) / 128;
  if (int(blockIdx.x) >= n_qt) return;  // shorter than the longest query sequence: no rows here
  // Query tiles with more live keys first (causal / right-bounded windows).
  const int qt = (p.wr >= 0) ? (n_qt - 1 - int(blockIdx.x)) : int(blockIdx.x);
  const int row0 = qt * 128;
  const int last_row = min(Sq, row0 + 128) - 1;
  const int kv_lo = live_range(row0, Sq, Sk, p.wl, p.wr).lo;
  const int kv_hi = live_range(last_row, Sq, Sk, p.wl, p.wr).hi;
  const int jb = kv_lo / 128;
  const int n_blocks = (kv_hi >= kv_lo) ? (kv_hi / 128 + 1 - jb) : 0;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::NK; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < C::NV; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, C::NCT / 32);  // one arrive per compute warp
    for (int s = 0; s < C::NDP; ++s) {
      mbar_init(&bars->dp_full[s], 1);
      mbar_init(&bars->ds_ready[s], C::NCT / 32);
    }
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->fac_ready, 1);
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
      tma_prefetch_desc_w(&tm_k);
      tma_prefetch_desc_w(&tm_v);
      tma_prefetch_desc_w(&tm_do);
      mbar_arrive_expect_tx_w(&bars->q_full, 2 * C::TILE_BYTES);
      for (int pn = 0; pn < C::PANELS; ++pn) {
        tma_load_4d_w(smem + C::Q_OFF + pn * C::PANEL_BYTES, &tm_q, &bars->q_full, pn * 64, h, sq_.q_off + row0,
                    sq_.tb);
        tma_load_4d_w(smem + C::DO_OFF + pn * C::PANEL_BYTES, &tm_do, &bars->q_full, pn * 64, h, sq_.q_off + row0,
                    sq_.tb);
      }
      int k_issued = 0, v_issued = 0;
      for (int jj = 0; jj < n_blocks; ++jj) {
        const int row = sq_.k_off + (jb + jj) * 128;
        const int sk = jj % C::NK, sv = jj % C::NV;
        if (!fa_wait_warp(&bars->k_empty[sk], (uint32_t(jj / C::NK) & 1u) ^ 1u, watch, SITE_DQ_EMPTY)) break;
        if (!(p.inject == FA_INJECT_BWD_SKIP_K && jj == 1)) {  // diagnostics: key tile 1 never arrives
          mbar_arrive_expect_tx_w(&bars->k_full[sk], C::TILE_BYTES);
          for (int pn = 0; pn < C::PANELS; ++pn)
            tma_load_4d_w(smem + C::K_OFF + sk * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_k, &bars->k_full[sk],
                          pn * 64, hkv, row, sq_.tb);
        }
        k_issued = jj + 1;
        if (!fa_wait_warp(&bars->v_empty[sv], (uint32_t(jj / C::NV) & 1u) ^ 1u, watch, SITE_DQ_EMPTY)) break;
        mbar_arrive_expect_tx_w(&bars->v_full[sv], C::TILE_BYTES);
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d_w(smem + C::V_OFF + sv * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_v, &bars->v_full[sv],
                        pn * 64, hkv, row, sq_.tb);
        v_issued = jj + 1;
      }
      drain_wait_b(&bars->q_full, 0, p.wait_ns);
      for (int jj = (k_issued > C::NK ? k_issued - C::NK : 0); jj < k_issued; ++jj)
        drain_wait_b(&bars->k_full[jj % C::NK], uint32_t(jj / C::NK) & 1u, p.wait_ns);
      for (int jj = (v_issued > C::NV ? v_issued - C::NV : 0); jj < v_issued; ++jj)
        drain_wait_b(&bars->v_full[jj % C::NV], uint32_t(jj / C::NV) & 1u, p.wait_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Per key tile jj: S(jj+1) as soon as every compute group holds S(jj) in
    // registers, then dP(jj+1) into the other dP buffer; both run while the
    // compute groups form dS(jj). Then dQ(jj) once dS(jj) is stored. dP(jj+2)
    // overwrites dS(jj) only after dQ(jj) has been issued (read in order).
    // Descriptors are built once per tile; each k-step is a constant added to
    // the start-address field.
    // The whole warp runs the loop; one elected lane issues each MMA and commit.
    if (n_blocks > 0) {
      constexpr uint32_t ID_SS = idesc_f16_f32(128, 128, 0, 0);  // S = Q K^T, dP = dO V^T
      constexpr uint32_t ID_DQ = idesc_f16_f32(128, D, 0, 1);    // dQ: dS from TMEM, K MN-major
      const uint64_t q_desc = sdesc_sw128(smem_u32(smem + C::Q_OFF), 16, 1024);
      const uint64_t do_desc = sdesc_sw128(smem_u32(smem + C::DO_OFF), 16, 1024);
      const uint64_t k_kdesc = sdesc_sw128(smem_u32(smem + C::K_OFF), 16, 1024);            // slot 0, K-major
      const uint64_t k_mdesc = sdesc_sw128(smem_u32(smem + C::K_OFF), C::PANEL_BYTES, 1024);  // slot 0, MN-major
      const uint64_t v_kdesc = sdesc_sw128(smem_u32(smem + C::V_OFF), 16, 1024);            // slot 0, K-major
      const uint32_t t_s = tmem + C::T_S, t_dp = tmem + C::T_DP, t_dq = tmem + C::T_DQ;
      auto issue_s = [&](int jj) {  // S(jj) = Q K_jj^T
        if (!fa_wait_warp(&bars->k_full[jj % C::NK], uint32_t(jj / C::NK) & 1u, watch, SITE_DQ_K)) return false;
        tc_fence_after();
        const uint64_t kd = sdesc_adv(k_kdesc, uint32_t(jj % C::NK) * C::TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::PANEL_BYTES + (kk % 4) * 32;
          mma_ss_w(t_s, sdesc_adv(q_desc, off), sdesc_adv(kd, off), ID_SS, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(&bars->s_full);
        return true;
      };
      auto issue_dp = [&](int jj) {  // dP(jj) = dO V_jj^T into buffer jj % NDP
        if (!fa_wait_warp(&bars->v_full[jj % C::NV], uint32_t(jj / C::NV) & 1u, watch, SITE_DQ_V)) return false;
        tc_fence_after();
        const uint64_t vd = sdesc_adv(v_kdesc, uint32_t(jj % C::NV) * C::TILE_BYTES);
        const uint32_t dst = t_dp + uint32_t(jj % C::NDP) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::PANEL_BYTES + (kk % 4) * 32;
          mma_ss_w(dst, sdesc_adv(do_desc, off), sdesc_adv(vd, off), ID_SS, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(&bars->dp_full[jj % C::NDP]);
        mma_commit_w(&bars->v_empty[jj % C::NV]);  // V_jj: only dP reads it
        return true;
      };
      bool ok = fa_wait_warp(&bars->q_full, 0, watch, SITE_DQ_Q) && issue_s(0) && issue_dp(0);
      for (int jj = 0; jj < n_blocks && ok; ++jj) {
        if (jj + 1 < n_blocks) {
          if (!(ok = fa_wait_warp(&bars->s_free, uint32_t(jj) & 1u, watch, SITE_DQ_S))) break;
          if (!(ok = issue_s(jj + 1) && issue_dp(jj + 1))) break;
        }
        // dQ += dS K ; keys 16kk..16kk+15 of dS sit at its buffer's columns 16kk+0..7
        const int pb = jj % C::NDP;
        if (!(ok = fa_wait_warp(&bars->ds_ready[pb], uint32_t(jj / C::NDP) & 1u, watch, SITE_DQ_DS))) break;
        tc_fence_after();
        {
          const uint64_t kd = sdesc_adv(k_mdesc, uint32_t(jj % C::NK) * C::TILE_BYTES);
          const uint32_t src = t_dp + uint32_t(pb) * 128;
          const uint32_t acc0 = jj > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts_w(t_dq, src + kk * 16, sdesc_adv(kd, kk * 2048), ID_DQ, kk > 0 ? 1u : acc0);
        }
        mma_commit_w(&bars->k_empty[jj % C::NK]);  // K_jj: read by S_jj and this dQ
      }
      if (ok) {
        mma_commit_w(&bars->acc_done);
      } else {
        mma_commit_w(&bars->drain);
        drain_wait_b(&bars->drain, 0, p.wait_ns);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ range factors of the group
    if (lane == 0) {
      const GroupExp ge = group_exps(p.amax, b, hkv, p.Hk);
      bars->fac[0] = p.scale_log2 * pow2f(-ge.q) * pow2f(-ge.k);
      unscale_factors(p.scale, ge.dO + ge.v + ge.k, bars->fac[1], bars->fac[2]);
      mbar_arrive(&bars->fac_ready);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ compute (thread = query row)
    const int w = (warp - 4) / 4;  // key-column group: columns [w*COLS, (w+1)*COLS)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int i = row0 + r;
    const uint32_t lane_addr = uint32_t(wq * 32) << 16;
    const RowRange rr = live_range(i, Sq, Sk, p.wl, p.wr);
    const int tile_lo_max = live_range(last_row, Sq, Sk, p.wl, p.wr).lo;
    const int tile_hi_min = live_range(row0, Sq, Sk, p.wl, p.wr).hi;
    const size_t vi = (size_t(b) * p.H + h) * p.Sq_pad + i;  // i < Sq_pad always
    const float nl2 = p.nl2[vi];
    const float dval = p.dvec[vi];
    const bool has_alibi = p.alibi != nullptr;
    const float slope_log2 = has_alibi ? p.alibi[b * p.alibi_bstride + h] * 1.4426950408889634f : 0.0f;
    const int c_i = i + Sk - Sq;
    // the group's range factors (warp 2): S arrives as 2^(eq+ek) S
    bool ok = fa_wait_warp(&bars->fac_ready, 0, watch, SITE_DQ_FAC);
    const float sl = bars->fac[0];
    for (int jj = 0; jj < n_blocks && ok; ++jj) {
      const int kb = (jb + jj) * 128 + w * C::COLS;  // first key of this group
      if (!(ok = fa_wait_warp(&bars->s_full, uint32_t(jj) & 1u, watch, SITE_DQ_S))) break;
      tc_fence_after();
      float pv[C::COLS];
      tmem_ld_cols(tmem + lane_addr + C::T_S + w * C::COLS, pv);
      tc_fence_before();
      mbar_arrive_warp(&bars->s_free);
      const int kbase = (jb + jj) * 128;
      const bool need_mask = !(kbase >= tile_lo_max && kbase + 127 <= tile_hi_min);
      if (has_alibi && (kb + C::COLS - 1 <= c_i || kb >= c_i)) {
        // keys on one side of the diagonal: the bias on column pairs, with the
        // signed slope (same rounding as the scalar form below)
        const float d0 = float(c_i - kb);
        const float ns = (kb >= c_i) ? slope_log2 : -slope_log2;
        const uint64_t ns2 = f2_pack(ns, ns), sl2 = f2_pack(sl, sl), nl2p = f2_pack(nl2, nl2);
        const uint64_t st2 = f2_pack(4.0f, 4.0f);
        uint64_t dist[2] = {f2_pack(d0, d0 - 1.0f), f2_pack(d0 - 2.0f, d0 - 3.0f)};
#pragma unroll
        for (int c = 0; c < C::COLS; c += 4) {
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int cc = c + 2 * k;
            float a0, a1;
            f2_unpack(f2_fma(f2_pack(pv[cc], pv[cc + 1]), sl2, f2_add(f2_mul(dist[k], ns2), nl2p)), a0, a1);
            pv[cc] = ex2_approx(a0);
            pv[cc + 1] = ex2_approx(a1);
            dist[k] = f2_sub(dist[k], st2);
          }
        }
      } else if (has_alibi) {
        const float d0 = float(c_i - kb);
#pragma unroll
        for (int c = 0; c < C::COLS; ++c)
          pv[c] = ex2_approx(fmaf(pv[c], sl, -slope_log2 * fabsf(d0 - float(c)) + nl2));
      } else {
        const uint64_t sl2 = f2_pack(sl, sl), nl2p = f2_pack(nl2, nl2);
#pragma unroll
        for (int c = 0; c < C::COLS; c += 2) {
          float a0, a1;
          f2_unpack(f2_fma(f2_pack(pv[c], pv[c + 1]), sl2, nl2p), a0, a1);
          pv[c] = ex2_approx(a0);
          pv[c + 1] = ex2_approx(a1);
        }
      }
      if (need_mask) {
        const int lo = rr.lo - kb, hi = rr.hi - kb;
#pragma unroll
        for (int c = 0; c < C::COLS; ++c) pv[c] = (c >= lo && c <= hi) ? pv[c] : 0.0f;
      }
      const int pb = jj % C::NDP;
      if (!(ok = fa_wait_warp(&bars->dp_full[pb], uint32_t(jj / C::NDP) & 1u, watch, SITE_DQ_DP))) break;
      tc_fence_after();
      // per 16-key chunk: load dP, form dS, store it as fp16 pairs over the chunk's
      // consumed dP columns (see the TMEM map)
#pragma unroll
      for (int ch = 0; ch < C::COLS / 16; ++ch) {
        float dp[16];
        const uint32_t col = tmem + lane_addr + C::T_DP + uint32_t(pb) * 128 + w * C::COLS + 16 * ch;
        tmem_ld_cols(col, dp);
        uint32_t pk[8];
        uint32_t keep = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float s0, s1;
          if constexpr (DROP) {  // keys kb + c .. : one generator call per four keys
            const int c = 16 * ch + 2 * e;
            if ((e & 1) == 0) keep = dropout_keep4(p.drop, b * p.H + h, i, (kb + c) >> 2);
            const float z0 = (keep >> (c & 3)) & 1u ? p.drop.keep_scale : 0.0f;
            const float z1 = (keep >> ((c & 3) + 1)) & 1u ? p.drop.keep_scale : 0.0f;
            ds_pair(pv[16 * ch + 2 * e], pv[16 * ch + 2 * e + 1], dp[2 * e] * z0, dp[2 * e + 1] * z1, dval, dval, s0,
                    s1);
          } else {
            ds_pair(pv[16 * ch + 2 * e], pv[16 * ch + 2 * e + 1], dp[2 * e], dp[2 * e + 1], dval, dval, s0, s1);
          }
          pk[e] = pack_f16x2(s0, s1);
        }
        tmem_st_x8(col, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(&bars->ds_ready[pb]);
    }
    // ------------------------------------------------------------ dQ epilogue (each group D/NCW columns)
    constexpr int SLICE = D / C::NCW;  // 16 or 32
    const bool row_ok = i < Sq;
    const size_t qrow = p.cu_q ? size_t(sq_.q_off) + i : size_t(b) * Sq + i;
    __nv_bfloat16* dst = p.dq + (qrow * p.H + h) * size_t(D) + w * SLICE;
    if (n_blocks == 0) {
      if (row_ok)
        for (int e = 0; e < SLICE / 8; ++e) reinterpret_cast<uint4*>(dst)[e] = make_uint4(0, 0, 0, 0);
    } else if (ok && fa_wait_warp(&bars->acc_done, 0, watch, SITE_DQ_ACC)) {
      tc_fence_after();
      float a[SLICE];
      tmem_ld_cols(tmem + lane_addr + C::T_DQ + w * SLICE, a);
      if (row_ok) {
        uint32_t pk[SLICE / 2];
        const float mul = bars->fac[1], mul2 = bars->fac[2];  // dQ' = 2^(edo+ev+ek) dQ / scale
#pragma unroll
        for (int e = 0; e < SLICE / 2; ++e) pk[e] = pack_bf16x2(a[2 * e] * mul * mul2, a[2 * e + 1] * mul * mul2);
#pragma unroll
        for (int e = 0; e < SLICE / 8; ++e)
          reinterpret_cast<uint4*>(dst)[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
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

static size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace: L2 and D vectors (B, H, Sq_pad) fp32 (Sq_pad: the longest query
// sequence rounded up to 128 rows), then fp16 copies of Q, dO (rows_q tokens,
// H heads) and K, V (rows_k tokens, Hk heads), then the group maxima (B, Hk, 4)
// and their replicas (B, Hk, AMAX_REPS, 4) uint32, then (fused dQ only) the
// fp32 dQ accumulator (rows_q, H, D), each region 256-byte aligned.
struct BwdWs {
  size_t vec, qside, kside, amax, reps, dqa;
  size_t total() const { return 2 * vec + 2 * qside + 2 * kside + amax + reps + dqa; }
};
static BwdWs bwd_ws(int B, int max_sq, long long rows_q, long long rows_k, int H, int Hk, int D, bool fdq) {
  const size_t sq_pad = size_t((max_sq + 127) / 128) * 128;
  return BwdWs{al256(size_t(B) * H * sq_pad * 4), al256(size_t(rows_q) * H * D * 2),
               al256(size_t(rows_k) * Hk * D * 2), al256(size_t(B) * Hk * 16),
               al256(size_t(B) * Hk * AMAX_REPS * 16), fdq ? al256(size_t(rows_q) * H * D * 4) : 0};
}

// The fused dQ (dK/dV kernel plus TMA reductions of dQ) runs for D = 64 when
// the caller does not ask for bitwise reproducibility: the reductions' order
// varies from run to run.
static bool bwd_fused_dq(int D, int deterministic) { return D == 64 && !deterministic; }

size_t bwd_workspace_bytes(int B, int Sq, int Sk, int H, int Hk, int D, int deterministic) {
  return bwd_ws(B, Sq, (long long)B * Sq, (long long)B * Sk, H, Hk, D, bwd_fused_dq(D, deterministic)).total();
}

size_t bwd_varlen_workspace_bytes(int B, int total_q, int total_k, int max_sq, int H, int Hk, int D) {
  return bwd_ws(B, max_sq, total_q, total_k, H, Hk, D, false).total();
}

// dQ from the fused dK/dV kernel's fp32 accumulator (already unscaled) to bf16,
// eight values per thread; n8 = elements / 8.
__global__ void __launch_bounds__(256) fa_bwd_dq_convert_kernel(const float* __restrict__ acc,
                                                                 __nv_bfloat16* __restrict__ dq, long long n8) {
  for (long long t = blockIdx.x * 256LL + threadIdx.x; t < n8; t += (long long)gridDim.x * 256) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * t];
    const float4 c = reinterpret_cast<const float4*>(acc)[2 * t + 1];
    reinterpret_cast<uint4*>(dq)[t] =
        make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(c.x, c.y), pack_bf16x2(c.z, c.w));
  }
}

template <int D>
static int launch_bwd_t(const AttnShape& s, const void* dout, const void* q, const void* k, const void* v,
                        const void* out, const float* lse, void* dq, void* dk, void* dv, void* ws,
                        int deterministic, const VarlenArgs* vl, const Dropout* dr, cudaStream_t stream) {
  BwdParams p;
  p.B = s.B;
  p.Sq = s.Sq;
  p.Sk = s.Sk;
  p.H = s.H;
  p.Hk = s.Hk;
  p.group = s.H / s.Hk;
  p.Sq_pad = ((s.Sq + 127) / 128) * 128;
  p.n_qt = p.Sq_pad / 128;
  p.cu_q = vl ? vl->cu_q : nullptr;
  p.cu_k = vl ? vl->cu_k : nullptr;
  p.total_q = vl ? vl->total_q : 0;
  p.total_k = vl ? vl->total_k : 0;
  p.drop = dr ? *dr : Dropout{0, 1.0f, 0, 0, 0};
  const bool drop = p.drop.thr != 0;
  const long long rows_q = vl ? vl->total_q : (long long)s.B * s.Sq;
  const long long rows_k = vl ? vl->total_k : (long long)s.B * s.Sk;
  // the fused dQ for dense, dropout-free calls (the workspace of those has the accumulator)
  const bool fdq = bwd_fused_dq(D, deterministic) && !vl && !drop;
  const BwdWs L = bwd_ws(s.B, s.Sq, rows_q, rows_k, s.H, s.Hk, D, bwd_fused_dq(D, deterministic) && !vl);
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.nl2 = reinterpret_cast<float*>(w);
  p.dvec = reinterpret_cast<float*>(w + L.vec);
  p.q16 = reinterpret_cast<uint16_t*>(w + 2 * L.vec);
  p.do16 = reinterpret_cast<uint16_t*>(w + 2 * L.vec + L.qside);
  p.k16 = reinterpret_cast<uint16_t*>(w + 2 * L.vec + 2 * L.qside);
  p.v16 = reinterpret_cast<uint16_t*>(w + 2 * L.vec + 2 * L.qside + L.kside);
  p.amax = reinterpret_cast<uint32_t*>(w + 2 * L.vec + 2 * L.qside + 2 * L.kside);
  p.amax_rep = reinterpret_cast<uint32_t*>(w + 2 * L.vec + 2 * L.qside + 2 * L.kside + L.amax);
  p.n_chunks = (std::max(p.Sq_pad, s.Sk) + CHUNK_TOK - 1) / CHUNK_TOK;  // s.Sk: the longest key sequence
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.out = static_cast<const __nv_bfloat16*>(out);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
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
  p.status = device_status_word();
  {
    const DebugSettings dbg = debug_settings();
    p.wait_ns = dbg.wait_ns;
    p.inject = dbg.inject;
  }
  if (!p.status) return FA_ERR_CUDA;
  if (s.B > 65535 || s.H > 65535) return FA_ERR_UNSUPPORTED;
  // Packed sequences are one (1, total, H, D) tensor.
  const int mb = vl ? 1 : s.B;
  const int mq_rows = vl ? vl->total_q : s.Sq, mk_rows = vl ? vl->total_k : s.Sk;
  CUtensorMap mq, mk, mv, mdo;
  if (!make_bshd_map(&mq, p.q16, mb, mq_rows, s.H, D, 128, true) ||
      !make_bshd_map(&mk, p.k16, mb, mk_rows, s.Hk, D, 128, true) ||
      !make_bshd_map(&mv, p.v16, mb, mk_rows, s.Hk, D, 128, true) ||
      !make_bshd_map(&mdo, p.do16, mb, mq_rows, s.H, D, 128, true))
    return FA_ERR_CUDA;

  {
    // the replicas start at zero; the pre-pass raises them, then the rescale
    // pass folds them and redoes the copies of groups that need a range factor
    if (cudaMemsetAsync(p.amax_rep, 0, L.reps, stream) != cudaSuccess) return FA_ERR_CUDA;
    const long long cpr = D / 8;
    const long long n_q = (rows_q * s.H * cpr + 31) & ~31LL;
    const long long n_k = (rows_k * s.Hk * cpr + 31) & ~31LL;
    const long long total = n_q + n_k + (long long)s.B * s.H * p.Sq_pad;
    // as many blocks as fit on the GPU at once: the grid strides over the items
    static int per_sm[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FA_ERR_CUDA;
    if (per_sm[dev] == 0) {
      int n = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fa_bwd_pre_kernel<D>, 256, 0) != cudaSuccess || n < 1)
        n = 1;
      per_sm[dev] = n;
    }
    const long long cap = (long long)device_sm_count() * per_sm[dev];
    fa_bwd_pre_kernel<D><<<int(std::max(1LL, std::min(cap, (total + 255) / 256))), 256, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    // about two blocks per SM over all groups, at least one per group
    const long long groups = (long long)s.B * s.Hk;
    const int rx = int(std::max(1LL, std::min((long long)p.n_chunks, (2LL * device_sm_count() + groups - 1) / groups)));
    fa_bwd_rescale_kernel<D><<<dim3(rx, s.Hk, s.B), 256, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  }
  const dim3 kv_grid((s.Sk + 127) / 128, s.Hk, s.B);
  if constexpr (D == 64) {
    if (fdq) {
      // dK/dV kernel with the dQ shares added into the zeroed accumulator, then bf16
      float* dqa = reinterpret_cast<float*>(w + 2 * L.vec + 2 * L.qside + 2 * L.kside + L.amax + L.reps);
      using CF = KvCfg<D, true>;
      CUtensorMap mdqa;
      if (!make_bshd_map_f32(&mdqa, dqa, s.B, s.Sq, s.H, D, CF::DQC, 32)) return FA_ERR_CUDA;  // one warp's box
      if (cudaMemsetAsync(dqa, 0, size_t(rows_q) * s.H * D * 4, stream) != cudaSuccess) return FA_ERR_CUDA;
      auto kf = fa_bwd_dkdv_kernel<D, false, true>;
      if (cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM_BYTES) != cudaSuccess)
        return FA_ERR_CUDA;
      kf<<<kv_grid, CF::THREADS, CF::SMEM_BYTES, stream>>>(mq, mk, mv, mdo, mdqa, p);
      if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
      const long long n8 = rows_q * s.H * D / 8;
      const long long cgrid = std::max(1LL, std::min((long long)device_sm_count() * 8, (n8 + 255) / 256));
      fa_bwd_dq_convert_kernel<<<unsigned(cgrid), 256, 0, stream>>>(dqa, p.dq, n8);
      return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
    }
  }
  auto kv = drop ? fa_bwd_dkdv_kernel<D, true, false> : fa_bwd_dkdv_kernel<D, false, false>;
  if (cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, KvCfg<D>::SMEM_BYTES) != cudaSuccess)
    return FA_ERR_CUDA;
  kv<<<kv_grid, KvCfg<D>::THREADS, KvCfg<D>::SMEM_BYTES, stream>>>(mq, mk, mv, mdo, mq, p);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  auto dqk = drop ? fa_bwd_dq_kernel<D, true> : fa_bwd_dq_kernel<D, false>;
  if (cudaFuncSetAttribute(dqk, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::SMEM_BYTES) != cudaSuccess)
    return FA_ERR_CUDA;
  dqk<<<dim3(p.n_qt, s.H, s.B), DqCfg<D>::THREADS, DqCfg<D>::SMEM_BYTES, stream>>>(mq, mk, mv, mdo, p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int bwd_launch(const AttnShape& s, const void* dout, const void* q, const void* k, const void* v, const void* out,
               const float* lse, void* dq, void* dk, void* dv, void* workspace, int deterministic,
               const VarlenArgs* varlen, const Dropout* dropout, cudaStream_t stream) {
  switch (s.D) {
    case 64:
      return launch_bwd_t<64>(s, dout, q, k, v, out, lse, dq, dk, dv, workspace, deterministic, varlen, dropout,
                              stream);
    case 128:
      return launch_bwd_t<128>(s, dout, q, k, v, out, lse, dq, dk, dv, workspace, deterministic, varlen, dropout,
                               stream);
    default:
      return FA_ERR_UNSUPPORTED;
  }
}

}  // namespace fa
