// Split-KV decode for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run decode: code that must not allocate inside a latency-critical or
// pre-planned region, runtimes whose memory is owned by another allocator,
// or hosts that forbid allocation after start-up. fa_decode_splitkv needs a
// caller-provided workspace for its per-split partial results; this entry
// point instead keeps them in a fixed array of the library's own device
// memory (g_decode_scratch below), so the caller passes only inputs and
// outputs.
//
// Rules of use:
//  * The array holds kScratchBytes on every GPU that loads the library, for
//    the life of the process. Requests whose partials would not fit
//    (fa_decode_workspace_size() > kScratchBytes) are rejected with
//    FA_ERR_WORKSPACE.
//  * Its device address is looked up once per device, on the first call
//    made with that device current; make that first call before any stream
//    capture.
//  * Every call shares the one array. Calls whose kernels overlap on the GPU
//    (different streams, or different host threads) race on it; order them.
//  * Nothing in it needs to start at zero: every partial slot a call reads is
//    written by the same call first, so leftovers of earlier calls are harmless.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/fa.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;  // 8 MiB of split partials
constexpr int kMaxDev = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

// Device address of g_decode_scratch on the current device. In host code the
// symbol itself is only a host-side handle, never a usable device address.
void* scratch_address() {
  static void* ptrs[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int fa_decode_splitkv_noalloc(const void* q, const void* k_cache, const void* v_cache, void* out,
                                         float* lse, int B, int Sq, int Sk, int H, int Hk, int D, float scale,
                                         int causal, int window_left, int window_right, const float* alibi_slopes,
                                         int alibi_batch_stride, int num_splits, fa_stream_t stream) {
  if (!q || !k_cache || !v_cache || !out || !lse) return FA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(lse))
    return FA_ERR_INVALID;
  if (B < 1 || Sq < 1 || Sk < 1 || H < 1 || D < 1) return FA_ERR_INVALID;
  if (Hk < 1 || H % Hk != 0) return FA_ERR_INVALID;
  if (window_left < -1 || window_right < -1) return FA_ERR_INVALID;
  if (alibi_slopes) {
    if (reinterpret_cast<uintptr_t>(alibi_slopes) & 3u) return FA_ERR_INVALID;
    if (alibi_batch_stride != 0 && alibi_batch_stride != H) return FA_ERR_INVALID;
  }
  if (Sq > 16 || Sk > (1 << 30)) return FA_ERR_UNSUPPORTED;
  if (B > 65535 || H > 65535) return FA_ERR_UNSUPPORTED;  // gridDim.y and gridDim.z limits
  if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
  if (num_splits < 0 || num_splits > 256) return FA_ERR_INVALID;
  const int n = num_splits == 0 ? fa::decode_auto_splits(B, Sq, Sk, H, Hk, D) : num_splits;
  if (fa::decode_workspace_bytes(B, Sq, H, D, n) > kScratchBytes) return FA_ERR_WORKSPACE;
  void* ws = scratch_address();
  if (!ws) return FA_ERR_CUDA;
  fa::AttnShape s;
  s.B = B;
  s.Sq = Sq;
  s.Sk = Sk;
  s.H = H;
  s.Hk = Hk;
  s.D = D;
  s.scale = (scale > 0.0f && isfinite(scale)) ? scale : 1.0f / sqrtf(float(D));
  s.wl = window_left;
  s.wr = causal ? 0 : window_right;
  s.alibi = alibi_slopes;
  s.alibi_bstride = alibi_slopes ? alibi_batch_stride : 0;
  return fa::decode_launch(s, q, k_cache, v_cache, out, lse, ws, n, nullptr, reinterpret_cast<cudaStream_t>(stream));
}
