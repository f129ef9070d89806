// Host-side declarations shared by the C-ABI layer and the kernel launchers.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "philox.cuh"
#include "rotary.cuh"

namespace fa {

// Arguments common to every attention entry point, after validation.
struct AttnShape {
  int B, Sq, Sk, H, D;
  int Hk;             // key/value heads; H is a multiple of Hk, query head h reads kv head h / (H / Hk)
  float scale;        // softmax scale (already defaulted)
  int wl, wr;         // window, causal folded into wr (= 0); -1 unbounded
  const float* alibi; // NULL or fp32 slopes
  int alibi_bstride;  // 0 (slopes (H,)) or H (slopes (B,H))
};

// Packed sequences: cumulative lengths cu_q, cu_k (device int32, B + 1 each,
// starting at 0) and the packed row counts. With these the kernels take each
// sequence's own lengths and rows; AttnShape's Sq, Sk are the longest ones.
struct VarlenArgs {
  const int* cu_q;
  const int* cu_k;
  int total_q, total_k;
};

// Decode over a cache with per-sequence lengths: dense (B, cap, Hk, D) caches
// (block_table NULL) or pages (num_pages, page_size, Hk, D), key block p of
// sequence b in page block_table[b * max_pages + p]. Sequence b has
// min(seqlens[b] + s_new, cap) keys, the last s_new appended in this call.
// rot: rotary embedding of q (and of the appended keys); rot.cos NULL for none.
struct CacheArgs {
  const int* block_table;
  const int* seqlens;
  int num_pages, page_size, max_pages;
  int s_new, cap;
  Rotary rot;
};

// Argument checks shared by every attention entry point: sizes, head groups,
// window bounds, ALiBi pointer and stride, and the grid limits (B, H <= 65535,
// Sq, Sk <= 2^30). Fills `s` with the defaults folded in (scale <= 0 or NaN ->
// 1/sqrt(D), causal -> window right = 0). Returns FA_OK or a negative fa_status;
// the supported head dims are checked by each caller.
int check_common(int B, int Sq, int Sk, int H, int Hk, int D, float scale, int causal, int wl, int wr,
                 const float* alibi, int alibi_bstride, AttnShape* s);

// Diagnostic settings the launchers pass to the kernels: the bounded-wait
// limit (FA_WAIT_TIMEOUT_NS) and a fault to inject (FA_INJECT_NONE), both
// process-wide and changed only by fa_debug_set_fault().
struct DebugSettings {
  uint64_t wait_ns;
  unsigned int inject;
};
DebugSettings debug_settings();

// Status word of the current device (device pointer), or NULL on failure.
unsigned int* device_status_word();

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Encodes a 4-D tiled TMA map over a (B, S, H, D) 16-bit tensor (bf16, or
// fp16 with `f16` set): box of 64 head-dim elements (128 B, 128-byte swizzle)
// x 1 head x `box_rows` rows x 1 batch. Returns false if the driver rejects it.
bool make_bshd_map(CUtensorMap* map, const void* base, int B, int S, int H, int D, int box_rows, bool f16 = false);
// As make_bshd_map with a box of box_heads consecutive heads x box_rows rows
// (smem rows ordered row-major over (row, head)).
bool make_bshd_map_box(CUtensorMap* map, const void* base, int B, int S, int H, int D, int box_heads, int box_rows,
                       bool f16 = false);
// fp32 (B, S, H, D) tensor in boxes of box_cols columns x box_rows rows of one
// head, for TMA reductions; rows of box_cols * 4 = 64 bytes take the 64-byte
// swizzle, rows of 128 bytes the 128-byte swizzle.
bool make_bshd_map_f32(CUtensorMap* map, const void* base, int B, int S, int H, int D, int box_cols, int box_rows);

// Kernel launchers (return an fa_status value).
int fwd_launch(const AttnShape& s, const void* q, const void* k, const void* v, void* out, float* lse,
               const VarlenArgs* varlen, const Dropout* dropout, cudaStream_t stream);
int decode_launch(const AttnShape& s, const void* q, const void* k, const void* v, void* out, float* lse,
                  void* workspace, int num_splits, const CacheArgs* cache, cudaStream_t stream);
// Writes the s_new rows of k_new, v_new (B, s_new, Hk, D) into the cache behind
// seqlens[b], the keys rotated (cache.rot); run before decode_launch.
int kv_append_launch(const AttnShape& s, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                     const CacheArgs& cache, cudaStream_t stream);
// Workspace of a decode call: the split partials, then (with_rotary) the rotated
// query pair that only a rotary call on the tensor-core kernel writes.
size_t decode_workspace_bytes(int B, int Sq, int H, int D, int num_splits, bool with_rotary = true);
// FA_ERR_UNSUPPORTED when the split kernel's grid would exceed the hardware's
// limits; checked before the first launch of a decode call.
int decode_check(const AttnShape& s, const CacheArgs* cache);
int decode_auto_splits(int B, int Sq, int Sk, int H, int Hk, int D);
int bwd_launch(const AttnShape& s, const void* dout, const void* q, const void* k, const void* v,
               const void* out, const float* lse, void* dq, void* dk, void* dv, void* workspace,
               int deterministic, const VarlenArgs* varlen, const Dropout* dropout, cudaStream_t stream);
size_t bwd_varlen_workspace_bytes(int B, int total_q, int total_k, int max_sq, int H, int Hk, int D);
size_t bwd_workspace_bytes(int B, int Sq, int Sk, int H, int Hk, int D, int deterministic);

}  // namespace fa
