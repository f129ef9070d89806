// C-ABI entry points of libfa_gb300.so (declared in include/fa.h).
//
// This layer validates arguments, folds the defaults (scale = 1/sqrt(D),
// causal => window_right = 0), and hands a validated AttnShape to the kernel
// launchers. It allocates nothing: all tensors and workspaces belong to the
// caller. The one piece of library state is a device status word per GPU
// (a __device__ variable), which bounded waits inside the kernels set.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/fa.h"
#include "fa_device.cuh"
#include "internal.h"

namespace fa {

__device__ unsigned int g_status_word;

static constexpr int kMaxDevices = 64;

static std::atomic<uint64_t> g_wait_ns{FA_WAIT_TIMEOUT_NS};
static std::atomic<unsigned int> g_inject{FA_INJECT_NONE};

DebugSettings debug_settings() { return DebugSettings{g_wait_ns.load(), g_inject.load()}; }

unsigned int* device_status_word() {
  static unsigned int* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned int*>(p);
  }
  return ptrs[dev];
}

int device_sm_count() {
  static int counts[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  if (counts[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    counts[dev] = n;
  }
  return counts[dev];
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_bshd_map(CUtensorMap* map, const void* base, int B, int S, int H, int D, int box_rows, bool f16) {
  return make_bshd_map_box(map, base, B, S, H, D, 1, box_rows, f16);
}

bool make_bshd_map_box(CUtensorMap* map, const void* base, int B, int S, int H, int D, int box_heads, int box_rows,
                       bool f16) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {cuuint64_t(D), cuuint64_t(H), cuuint64_t(S), cuuint64_t(B)};
  cuuint64_t strides[3] = {cuuint64_t(D) * 2, cuuint64_t(H) * D * 2, cuuint64_t(S) * H * D * 2};
  cuuint32_t box[4] = {64, cuuint32_t(box_heads), cuuint32_t(box_rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_bshd_map_f32(CUtensorMap* map, const void* base, int B, int S, int H, int D, int box_cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {cuuint64_t(D), cuuint64_t(H), cuuint64_t(S), cuuint64_t(B)};
  cuuint64_t strides[3] = {cuuint64_t(D) * 4, cuuint64_t(H) * D * 4, cuuint64_t(S) * H * D * 4};
  cuuint32_t box[4] = {cuuint32_t(box_cols), 1, cuuint32_t(box_rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, box_cols * 4 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int check_common(int B, int Sq, int Sk, int H, int Hk, int D, float scale, int causal, int wl, int wr,
                        const float* alibi, int alibi_bstride, AttnShape* s) {
  if (B < 1 || Sq < 1 || Sk < 1 || H < 1 || D < 1) return FA_ERR_INVALID;
  if (Hk < 1 || H % Hk != 0) return FA_ERR_INVALID;
  if (wl < -1 || wr < -1) return FA_ERR_INVALID;
  if (alibi) {
    if (reinterpret_cast<uintptr_t>(alibi) & 3u) return FA_ERR_INVALID;
    if (alibi_bstride != 0 && alibi_bstride != H) return FA_ERR_INVALID;
  }
  // Index ranges: rows and tiles are addressed with 32-bit ints, elements with 64-bit offsets.
  if (Sq > (1 << 30) || Sk > (1 << 30)) return FA_ERR_UNSUPPORTED;
  // Heads and batches index gridDim.y and gridDim.z, which allow at most 65535.
  if (B > 65535 || H > 65535) return FA_ERR_UNSUPPORTED;
  s->B = B;
  s->Sq = Sq;
  s->Sk = Sk;
  s->H = H;
  s->Hk = Hk;
  s->D = D;
  s->scale = (scale > 0.0f && isfinite(scale)) ? scale : 1.0f / sqrtf(float(D));
  s->wl = wl;
  s->wr = causal ? 0 : wr;
  s->alibi = alibi;
  s->alibi_bstride = alibi ? alibi_bstride : 0;
  return FA_OK;
}

}  // namespace fa

using fa::AttnShape;
using fa::check_common;

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

extern "C" {

int fa_version(void) { return 10000; }

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK:
      return "ok";
    case FA_ERR_INVALID:
      return "invalid argument";
    case FA_ERR_UNSUPPORTED:
      return "unsupported configuration";
    case FA_ERR_CUDA:
      return "CUDA runtime or driver error";
    case FA_ERR_TIMEOUT:
      return "device-side bounded wait expired";
    case FA_ERR_WORKSPACE:
      return "workspace missing, misaligned or too small";
    default:
      return "unknown status";
  }
}

int fa_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Sq, int Sk, int H, int Hk,
           int D, float scale, int causal, int window_left, int window_right, const float* alibi_slopes,
           int alibi_batch_stride, fa_stream_t stream) {
  if (!q || !k || !v || !out || !lse) return FA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse)) return FA_ERR_INVALID;
  AttnShape s;
  int st = check_common(B, Sq, Sk, H, Hk, D, scale, causal, window_left, window_right, alibi_slopes,
                        alibi_batch_stride, &s);
  if (st != FA_OK) return st;
  if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
  return fa::fwd_launch(s, q, k, v, out, lse, nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int fa_fwd_varlen(const void* q, const void* k, const void* v, void* out, float* lse, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int B, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                  int H, int Hk, int D, float scale, int causal, int window_left, int window_right,
                  const float* alibi_slopes, int alibi_batch_stride, fa_stream_t stream) {
  if (!q || !k || !v || !out || !lse || !cu_seqlens_q || !cu_seqlens_k) return FA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse)) return FA_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) || (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u))
    return FA_ERR_INVALID;
  if (total_q < 1 || total_k < 1) return FA_ERR_INVALID;
  AttnShape s;
  int st = check_common(B, max_seqlen_q, max_seqlen_k, H, Hk, D, scale, causal, window_left, window_right,
                        alibi_slopes, alibi_batch_stride, &s);
  if (st != FA_OK) return st;
  if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
  if (total_q > (1 << 30) || total_k > (1 << 30)) return FA_ERR_UNSUPPORTED;
  const fa::VarlenArgs vl{cu_seqlens_q, cu_seqlens_k, total_q, total_k};
  return fa::fwd_launch(s, q, k, v, out, lse, &vl, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

// Dropout rule shared by fa_fwd_dropout and fa_bwd_dropout; p in [0, 1).
static bool make_dropout(float p, uint64_t seed, uint32_t offset, fa::Dropout* d) {
  if (!(p >= 0.0f && p < 1.0f)) return false;
  const double t = double(p) * 4294967296.0;
  d->thr = t >= 4294967295.0 ? 4294967295u : uint32_t(t);
  d->keep_scale = 1.0f / (1.0f - p);
  d->seed_lo = uint32_t(seed);
  d->seed_hi = uint32_t(seed >> 32);
  d->offset = offset;
  return true;
}

int fa_fwd_dropout(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Sq, int Sk, int H,
                   int Hk, int D, float scale, int causal, int window_left, int window_right, const float* alibi_slopes,
                   int alibi_batch_stride, float dropout_p, uint64_t seed, uint32_t offset, fa_stream_t stream) {
  if (!q || !k || !v || !out || !lse) return FA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse)) return FA_ERR_INVALID;
  AttnShape s;
  int st = check_common(B, Sq, Sk, H, Hk, D, scale, causal, window_left, window_right, alibi_slopes,
                        alibi_batch_stride, &s);
  if (st != FA_OK) return st;
  if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
  fa::Dropout dr;
  if (!make_dropout(dropout_p, seed, offset, &dr)) return FA_ERR_INVALID;
  return fa::fwd_launch(s, q, k, v, out, lse, nullptr, &dr, reinterpret_cast<cudaStream_t>(stream));
}

int fa_bwd_dropout(const void* dout, const void* q, const void* k, const void* v, const void* out, const float* lse,
                   void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Sq, int Sk,
                   int H, int Hk, int D, float scale, int causal, int window_left, int window_right,
                   const float* alibi_slopes, int alibi_batch_stride, int deterministic, float dropout_p,
                   uint64_t seed, uint32_t offset, fa_stream_t stream) {
  if (!dout || !q || !k || !v || !out || !lse || !dq || !dk || !dv) return FA_ERR_INVALID;
  if (!aligned16(dout) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID;
  AttnShape s;
  int st = check_common(B, Sq, Sk, H, Hk, D, scale, causal, window_left, window_right, alibi_slopes,
                        alibi_batch_stride, &s);
  if (st != FA_OK) return st;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  fa::Dropout dr;
  if (!make_dropout(dropout_p, seed, offset, &dr)) return FA_ERR_INVALID;
  const size_t need = fa::bwd_workspace_bytes(B, Sq, Sk, H, Hk, D, deterministic);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return FA_ERR_WORKSPACE;
  return fa::bwd_launch(s, dout, q, k, v, out, lse, dq, dk, dv, workspace, deterministic, nullptr, &dr,
                        reinterpret_cast<cudaStream_t>(stream));
}

size_t fa_bwd_workspace_size(int B, int Sq, int Sk, int H, int Hk, int D, int deterministic) {
  if (B < 1 || Sq < 1 || Sk < 1 || H < 1 || Hk < 1 || H % Hk != 0 || (D != 64 && D != 128)) return 0;
  return fa::bwd_workspace_bytes(B, Sq, Sk, H, Hk, D, deterministic);
}

int fa_bwd(const void* dout, const void* q, const void* k, const void* v, const void* out, const float* lse,
           void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Sq, int Sk, int H,
           int Hk, int D, float scale, int causal, int window_left, int window_right, const float* alibi_slopes,
           int alibi_batch_stride, int deterministic, fa_stream_t stream) {
  if (!dout || !q || !k || !v || !out || !lse || !dq || !dk || !dv) return FA_ERR_INVALID;
  if (!aligned16(dout) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID;
  AttnShape s;
  int st = check_common(B, Sq, Sk, H, Hk, D, scale, causal, window_left, window_right, alibi_slopes,
                        alibi_batch_stride, &s);
  if (st != FA_OK) return st;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  const size_t need = fa::bwd_workspace_bytes(B, Sq, Sk, H, Hk, D, deterministic);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return FA_ERR_WORKSPACE;
  return fa::bwd_launch(s, dout, q, k, v, out, lse, dq, dk, dv, workspace, deterministic, nullptr, nullptr,
                        reinterpret_cast<cudaStream_t>(stream));
}

size_t fa_bwd_varlen_workspace_size(int B, int total_q, int total_k, int max_seqlen_q, int H, int Hk, int D) {
  if (B < 1 || total_q < 1 || total_k < 1 || max_seqlen_q < 1 || H < 1 || Hk < 1 || H % Hk != 0) return 0;
  if (D != 64 && D != 128) return 0;
  return fa::bwd_varlen_workspace_bytes(B, total_q, total_k, max_seqlen_q, H, Hk, D);
}

int fa_bwd_varlen(const void* dout, const void* q, const void* k, const void* v, const void* out, const float* lse,
                  void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int B, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                  int H, int Hk, int D, float scale, int causal, int window_left, int window_right,
                  const float* alibi_slopes, int alibi_batch_stride, int deterministic, fa_stream_t stream) {
  if (!dout || !q || !k || !v || !out || !lse || !dq || !dk || !dv || !cu_seqlens_q || !cu_seqlens_k)
    return FA_ERR_INVALID;
  if (!aligned16(dout) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) || (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u))
    return FA_ERR_INVALID;
  if (total_q < 1 || total_k < 1) return FA_ERR_INVALID;
  AttnShape s;
  int st = check_common(B, max_seqlen_q, max_seqlen_k, H, Hk, D, scale, causal, window_left, window_right,
                        alibi_slopes, alibi_batch_stride, &s);
  if (st != FA_OK) return st;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (total_q > (1 << 30) || total_k > (1 << 30)) return FA_ERR_UNSUPPORTED;
  const size_t need = fa::bwd_varlen_workspace_bytes(B, total_q, total_k, max_seqlen_q, H, Hk, D);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return FA_ERR_WORKSPACE;
  const fa::VarlenArgs vl{cu_seqlens_q, cu_seqlens_k, total_q, total_k};
  return fa::bwd_launch(s, dout, q, k, v, out, lse, dq, dk, dv, workspace, deterministic, &vl, nullptr,
                        reinterpret_cast<cudaStream_t>(stream));
}

int fa_decode_num_splits(int B, int Sq, int Sk, int H, int Hk, int D) {
  if (B < 1 || Sq < 1 || Sk < 1 || H < 1 || Hk < 1 || H % Hk != 0) return 1;
  return fa::decode_auto_splits(B, Sq, Sk, H, Hk, D);
}

size_t fa_decode_workspace_size(int B, int Sq, int Sk, int H, int Hk, int D, int num_splits) {
  if (B < 1 || Sq < 1 || Sq > 16 || Sk < 1 || H < 1 || (D != 64 && D != 128 && D != 256)) return 0;
  if (Hk < 1 || H % Hk != 0) return 0;
  if (num_splits < 0 || num_splits > 256) return 0;
  const int n = num_splits == 0 ? fa::decode_auto_splits(B, Sq, Sk, H, Hk, D) : num_splits;
  return fa::decode_workspace_bytes(B, Sq, H, D, n);
}

int fa_decode_splitkv(const void* q, const void* k_cache, const void* v_cache, void* out, float* lse,
                      void* workspace, size_t workspace_bytes, int B, int Sq, int Sk, int H, int Hk, int D,
                      float scale, int causal, int window_left, int window_right, const float* alibi_slopes,
                      int alibi_batch_stride, int num_splits, fa_stream_t stream) {
  if (!q || !k_cache || !v_cache || !out || !lse) return FA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(lse))
    return FA_ERR_INVALID;
  AttnShape s;
  int st = check_common(B, Sq, Sk, H, Hk, D, scale, causal, window_left, window_right, alibi_slopes,
                        alibi_batch_stride, &s);
  if (st != FA_OK) return st;
  if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
  if (Sq > 16) return FA_ERR_UNSUPPORTED;
  if (num_splits < 0 || num_splits > 256) return FA_ERR_INVALID;
  const int n = num_splits == 0 ? fa::decode_auto_splits(B, Sq, Sk, H, Hk, D) : num_splits;
  const size_t need = fa::decode_workspace_bytes(B, Sq, H, D, n);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return FA_ERR_WORKSPACE;
  return fa::decode_launch(s, q, k_cache, v_cache, out, lse, workspace, n, nullptr,
                           reinterpret_cast<cudaStream_t>(stream));
}

int fa_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                    const int* seqlens_k, void* out, float* lse, void* workspace, size_t workspace_bytes, int B,
                    int Sq, int max_seqlen_k, int num_pages, int page_size, int max_pages_per_seq, int H, int Hk,
                    int D, float scale, int causal, int window_left, int window_right, const float* alibi_slopes,
                    int alibi_batch_stride, int num_splits, fa_stream_t stream) {
  if (!q || !k_pages || !v_pages || !block_table || !seqlens_k || !out || !lse) return FA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out) || !aligned16(lse))
    return FA_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seqlens_k) & 3u))
    return FA_ERR_INVALID;
  if (num_pages < 1 || page_size < 1 || max_pages_per_seq < 1) return FA_ERR_INVALID;
  AttnShape s;
  int st = check_common(B, Sq, max_seqlen_k, H, Hk, D, scale, causal, window_left, window_right, alibi_slopes,
                        alibi_batch_stride, &s);
  if (st != FA_OK) return st;
  if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
  if (Sq > 16 || page_size % 128 != 0 || (long long)max_pages_per_seq * page_size > (1 << 30))
    return FA_ERR_UNSUPPORTED;
  if (num_splits < 0 || num_splits > 256) return FA_ERR_INVALID;
  const int n = num_splits == 0 ? fa::decode_auto_splits(B, Sq, max_seqlen_k, H, Hk, D) : num_splits;
  const size_t need = fa::decode_workspace_bytes(B, Sq, H, D, n);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return FA_ERR_WORKSPACE;
  const fa::CacheArgs cg{block_table, seqlens_k, num_pages, page_size, max_pages_per_seq,
                         0, max_pages_per_seq * page_size, fa::Rotary{nullptr, nullptr, 0, 0, 0}};
  return fa::decode_launch(s, q, k_pages, v_pages, out, lse, workspace, n, &cg, reinterpret_cast<cudaStream_t>(stream));
}

int fa_decode_kvcache(const void* q, void* k_cache, void* v_cache, const int* cache_seqlens, const void* k_new,
                      const void* v_new, int S_new, const float* rotary_cos, const float* rotary_sin, int rotary_dim,
                      int rotary_len, int rotary_interleaved, const int* block_table, int num_pages, int page_size,
                      int max_pages_per_seq, void* out, float* lse, void* workspace, size_t workspace_bytes, int B,
                      int Sq, int cache_rows, int H, int Hk, int D, float scale, int causal, int window_left,
                      int window_right, const float* alibi_slopes, int alibi_batch_stride, int num_splits,
                      fa_stream_t stream) {
  if (!q || !k_cache || !v_cache || !cache_seqlens || !out || !lse) return FA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(lse))
    return FA_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(cache_seqlens) & 3u) return FA_ERR_INVALID;
  if (S_new < 0 || (S_new > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))))
    return FA_ERR_INVALID;
  if (rotary_cos || rotary_sin) {
    if (!rotary_cos || !rotary_sin || (reinterpret_cast<uintptr_t>(rotary_cos) & 3u) ||
        (reinterpret_cast<uintptr_t>(rotary_sin) & 3u) || rotary_len < 1)
      return FA_ERR_INVALID;
    if (rotary_dim < 16 || rotary_dim > D || rotary_dim % 16 != 0) return FA_ERR_UNSUPPORTED;
  }
  const bool paged = block_table != nullptr;
  if (paged) {
    if (reinterpret_cast<uintptr_t>(block_table) & 3u) return FA_ERR_INVALID;
    if (num_pages < 1 || page_size < 1 || max_pages_per_seq < 1) return FA_ERR_INVALID;
    if (page_size % 128 != 0 || (long long)max_pages_per_seq * page_size > (1 << 30)) return FA_ERR_UNSUPPORTED;
  } else if (cache_rows < 1) {
    return FA_ERR_INVALID;
  }
  const int cap = paged ? max_pages_per_seq * page_size : cache_rows;
  AttnShape s;
  int st = check_common(B, Sq, cap, H, Hk, D, scale, causal, window_left, window_right, alibi_slopes,
                        alibi_batch_stride, &s);
  if (st != FA_OK) return st;
  if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
  if (Sq > 16) return FA_ERR_UNSUPPORTED;
  if (num_splits < 0 || num_splits > 256) return FA_ERR_INVALID;
  const int n = num_splits == 0 ? fa::decode_auto_splits(B, Sq, cap, H, Hk, D) : num_splits;
  const size_t need = fa::decode_workspace_bytes(B, Sq, H, D, n);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return FA_ERR_WORKSPACE;
  const fa::CacheArgs cg{block_table, cache_seqlens, num_pages, page_size, max_pages_per_seq, S_new, cap,
                         fa::Rotary{rotary_cos, rotary_sin, rotary_dim, rotary_len, rotary_interleaved ? 1 : 0}};
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // nothing is appended to the cache by a call that cannot run its attention
  if ((st = fa::decode_check(s, &cg)) != FA_OK) return st;
  st = fa::kv_append_launch(s, k_new, v_new, k_cache, v_cache, cg, cs);
  if (st != FA_OK) return st;
  return fa::decode_launch(s, q, k_cache, v_cache, out, lse, workspace, n, &cg, cs);
}

int fa_debug_set_fault(int fault, uint64_t wait_limit_ns) {
  if (fault < FA_FAULT_NONE || fault > FA_FAULT_BWD_SKIP_KEY_TILE) return FA_ERR_INVALID;
  if (wait_limit_ns != 0 && (wait_limit_ns < 1000000ull || wait_limit_ns > fa::FA_WAIT_TIMEOUT_NS))
    return FA_ERR_INVALID;
  static_assert(FA_FAULT_FWD_SKIP_KEY_TILE == int(fa::FA_INJECT_FWD_SKIP_K) &&
                    FA_FAULT_BWD_SKIP_KEY_TILE == int(fa::FA_INJECT_BWD_SKIP_K),
                "fault codes");
  fa::g_wait_ns.store(wait_limit_ns ? wait_limit_ns : fa::FA_WAIT_TIMEOUT_NS);
  fa::g_inject.store(unsigned(fault));
  return FA_OK;
}

int fa_device_status(fa_stream_t stream, unsigned int* detail) {
  if (detail) *detail = 0;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  unsigned int word = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&word, fa::g_status_word, sizeof(word)) != cudaSuccess) return FA_ERR_CUDA;
  if (word && cudaMemcpyToSymbol(fa::g_status_word, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
  if (detail) *detail = word;
  return word ? FA_ERR_TIMEOUT : FA_OK;
}

}  // extern "C"
