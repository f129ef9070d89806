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
//    the life of the process. It holds only split partials,
//    B * Sq * H * splits * (D + 1) fp32 values (each part rounded up to 256
//    bytes). With num_splits == 0 the automatic split count is lowered until
//    they fit; a request that does not fit even so, or an explicit
//    num_splits whose partials do not fit, is rejected with FA_ERR_WORKSPACE.
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
  fa::AttnShape s;
  const int st = fa::check_common(B, Sq, Sk, H, Hk, D, scale, causal, window_left, window_right, alibi_slopes,
                                  alibi_batch_stride, &s);
  if (st != FA_OK) return st;
  if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
  if (Sq > 16) return FA_ERR_UNSUPPORTED;
  if (num_splits < 0 || num_splits > 256) return FA_ERR_INVALID;
  // This call never runs rotary, so the array holds only the split partials.
  auto fits = [&](int n) { return fa::decode_workspace_bytes(B, Sq, H, D, n, false) <= kScratchBytes; };
  int n = num_splits;
  if (n == 0) {
    // the automatic count, lowered until its partials fit the array
    n = fa::decode_auto_splits(B, Sq, Sk, H, Hk, D);
    while (n > 1 && !fits(n)) --n;
  }
  if (!fits(n)) return FA_ERR_WORKSPACE;
  void* ws = scratch_address();
  if (!ws) return FA_ERR_CUDA;
  return fa::decode_launch(s, q, k_cache, v_cache, out, lse, ws, n, nullptr, reinterpret_cast<cudaStream_t>(stream));
}
