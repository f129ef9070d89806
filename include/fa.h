/*
 * fa.h — C ABI of the GB300 (sm_103a) exact-attention library, libfa_gb300.so.
 *
 * The library computes exact scaled dot-product attention,
 *     O = softmax(scale * Q K^T + bias, masked) V,
 * as defined on the page "FlashAttention：快速且内存高效的准确注意力机制"
 * (cloud.tencent.com.cn/developer/article/2433927), sections "使用示例" and
 * "参数说明" (arguments softmax_scale, causal, window_size, alibi_slopes,
 * deterministic). Section names below refer to that page.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor pointer is DEVICE memory owned by the caller, contiguous,
 *   16-byte aligned. The library never allocates, frees or keeps a pointer
 *   after the call returns.
 * - Layouts: q, out, dout, dq: (B, Sq, H, D) bf16; k, v, dk, dv, k_cache,
 *   v_cache: (B, Sk, Hk, D) bf16; lse: (B, H, Sq) fp32, natural-log row
 *   logsumexp of the masked, scaled scores.
 * - Hk is the number of key/value heads, 1 <= Hk, H a multiple of Hk. Query
 *   head h attends key/value head h / (H / Hk): grouped-query attention,
 *   Hk = 1 is multi-query and Hk = H plain multi-head. The page's
 *   FlashCrossAttention takes kv of shape (B, Sk, 2, H_k, D) (section
 *   "代码解读博客：FlashCrossAttention") without saying which query heads share
 *   a key/value head; consecutive groups of H / Hk is the reading taken.
 * - D (head dim) is 64, 128 or 256 (backward: 64 or 128).
 * - Size limits, FA_ERR_UNSUPPORTED beyond them: B and H at most 65535 (they
 *   index grid dimensions); Sq, Sk and the packed totals at most 2^30. Decode
 *   also refuses a call whose split grid (Hk x blocks of query pairs) exceeds
 *   65535 rows, or B * Sq * H above 2^31 - 1. It checks this before any
 *   launch, so a refused fa_decode_kvcache leaves the cache unchanged.
 * - scale <= 0 (or NaN) selects the default 1/sqrt(D) (section "参数说明").
 * - causal != 0 masks key j for query row i unless j <= i + Sk - Sq: the mask
 *   is aligned to the bottom-right corner of the score matrix (section
 *   "2.1：更改causal标志的行为").
 * - window_left / window_right >= 0 keep only keys j with
 *   i + Sk - Sq - window_left <= j <= i + Sk - Sq + window_right; -1 means
 *   unbounded on that side (sections "参数说明", "2.3：局部（即滑动窗口）注意力").
 *   causal != 0 forces window_right = 0.
 * - alibi_slopes: NULL, or fp32 device array of shape (H,) when
 *   alibi_batch_stride == 0, or (B, H) when alibi_batch_stride == H. The
 *   score of (i, j) gets -slope * |i + Sk - Sq - j| added after scaling
 *   (sections "参数说明", "2.4：ALiBi（线性偏差注意力），确定性反向传播").
 * - A query row with no live key gets O = 0 (section "2.1", last sentence)
 *   and lse = -inf.
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *   default stream). The return value reports argument checks and launch
 *   errors only. A kernel whose internal bounded wait expired records it in
 *   a device status word, read by fa_device_status().
 * - No entry point throws, exits or traps. Nothing falls back to another
 *   implementation.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fa_stream_t; /* same type as cudaStream_t */

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID = -1,     /* NULL/misaligned pointer, size < 1, bad window or ALiBi stride */
  FA_ERR_UNSUPPORTED = -2, /* valid request outside what is built (e.g. D = 96) */
  FA_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed (launch, tensor-map encode) */
  FA_ERR_TIMEOUT = -4,     /* a device-side bounded wait expired (from fa_device_status) */
  FA_ERR_WORKSPACE = -5    /* workspace pointer NULL/misaligned or workspace_bytes too small */
} fa_status;

/* Library version, major*10000 + minor*100 + patch. */
int fa_version(void);

/* Static description of a status code. Never NULL. */
const char* fa_status_string(int status);

/*
 * Forward. Writes out (B,Sq,H,D) bf16 and lse (B,H,Sq) fp32.
 * Computes, per (b, h), the tiled forward with an online softmax: for each
 * 128-row query tile the key/value tiles are streamed once, the running
 * output is kept unscaled and divided by the row sum only at the end, and
 * the row logsumexp L is saved for the backward (section "算法 / 前向传播").
 * Supported: D in {64, 128, 256}; any Sq, Sk >= 1.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Sq, int Sk, int H,
           int Hk, int D, float scale, int causal, int window_left, int window_right, const float* alibi_slopes,
           int alibi_batch_stride, fa_stream_t stream);

/*
 * Forward with dropout on the attention probabilities (section "参数说明":
 * dropout_p). The pages give no random generator; the one used here is
 * Philox4x32-10 (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3",
 * SC 2011). Entry (b, h, i, j) of the probability matrix P uses word j % 4 of
 * Philox4x32-10(counter = (j / 4, i, b * H + h, offset), key = (seed & 0xffffffff,
 * seed >> 32)); it is dropped when that word is below floor(dropout_p * 2^32)
 * and otherwise scaled by 1 / (1 - dropout_p). out = (P o Z) V; lse is that of
 * the undropped scores, as in fa_fwd. Same seed and offset give the same
 * mask in fa_bwd_dropout. Arguments otherwise as fa_fwd; 0 <= dropout_p < 1.
 */
int fa_fwd_dropout(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Sq, int Sk, int H,
                   int Hk, int D, float scale, int causal, int window_left, int window_right, const float* alibi_slopes,
                   int alibi_batch_stride, float dropout_p, uint64_t seed, uint32_t offset, fa_stream_t stream);

/*
 * Backward of fa_fwd_dropout with the same dropout_p, seed and offset:
 * dV = (P o Z)^T dO, dS = P o (Z o dO V^T - D), D_i = rowsum(dO o O),
 * dQ = scale dS K, dK = scale dS^T Q. Arguments otherwise as fa_bwd.
 */
int fa_bwd_dropout(const void* dout, const void* q, const void* k, const void* v, const void* out, const float* lse,
                   void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Sq, int Sk,
                   int H, int Hk, int D, float scale, int causal, int window_left, int window_right,
                   const float* alibi_slopes, int alibi_batch_stride, int deterministic, float dropout_p,
                   uint64_t seed, uint32_t offset, fa_stream_t stream);

/*
 * Forward over packed sequences of different lengths (page section
 * "代码解读博客：FlashSelfAttention": cu_seqlens, max_seqlen; the page's
 * flash_attn_varlen_func, section "函数重命名"). Sequence b has query rows
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of q (total_q, H, D) and key rows
 * cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1 of k, v (total_k, Hk, D); it is
 * attended exactly as fa_fwd would attend it alone (the causal diagonal and
 * the window are placed per sequence, ALiBi slopes are per b as in fa_fwd).
 * Writes out (total_q, H, D) bf16 and lse (H, total_q) fp32.
 * cu_seqlens_q, cu_seqlens_k: DEVICE int32 arrays of B + 1 non-decreasing
 * entries starting at 0 and ending at total_q / total_k (a sequence may be
 * empty). max_seqlen_q / max_seqlen_k must be at least the longest query /
 * key sequence: the grid is sized from them and rows beyond are not
 * computed. These arrays stay on the device and are not checked.
 */
int fa_fwd_varlen(const void* q, const void* k, const void* v, void* out, float* lse, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int B, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                  int H, int Hk, int D, float scale, int causal, int window_left, int window_right,
                  const float* alibi_slopes, int alibi_batch_stride, fa_stream_t stream);

/*
 * Bytes of device workspace fa_bwd needs: the per-row D_i = rowsum(dO * O)
 * and L*log2(e) vectors, (B, H, Sq rounded up to 128) fp32 each, fp16
 * copies of q, dout (B, Sq, H, D) and k, v (B, Sk, Hk, D), and the largest
 * magnitudes of q, k, v, dout per (batch, key/value head) group, (B, Hk, 4)
 * uint32 plus 32 replicas of them (B, Hk, 32, 4), and with D = 64 and
 * deterministic == 0 an fp32 dQ accumulator (B, Sq, H, D), each section
 * rounded up to 256 bytes. Returns 0 for arguments fa_bwd would reject.
 */
size_t fa_bwd_workspace_size(int B, int Sq, int Sk, int H, int Hk, int D, int deterministic);

/*
 * Backward (section "反向传播": recompute P from the saved logsumexp L, no
 * stored attention matrix). Inputs: dout, q, k, v, out (bf16) and lse (fp32)
 * from fa_fwd with the same arguments. Writes dq (B,Sq,H,D), dk, dv
 * (B,Sk,Hk,D) bf16; they are overwritten, not accumulated. With Hk < H the
 * dk and dv of a key/value head are the sums over the query heads sharing
 * it, formed inside one thread block.
 * deterministic (section "2.4": slower, bitwise reproducible): with 1 every
 * run is bitwise reproducible, because no output element is accumulated
 * across thread blocks: one kernel per 128-key tile produces dK and dV,
 * another per 128-row query tile produces dQ. With 0 and D = 64, the dK/dV
 * kernel also forms dQ and adds each 128-key tile's share into an fp32
 * accumulator in the workspace: dK and dV are the same bits as with 1, dQ
 * agrees to within its rounding but the order of its sums varies from run to
 * run. With 0 at D = 128 the two modes run the same kernels.
 * Precision: the products run on fp16 operands (copies of the inputs, P and
 * dS) with fp32 accumulation. Each (sequence, key/value head) group of q, k,
 * v and dout is copied times a power of two that puts its largest magnitude
 * in [4, 8) (or left as is when it lies in [1, 8)), and the factors are taken
 * back out exactly, so inputs of any finite bf16 magnitude keep fp16's
 * precision: gradients of 1e-8 are as accurate, relative to their size, as
 * gradients of 1. Non-finite inputs give non-finite gradients.
 * workspace: caller-owned device buffer of at least fa_bwd_workspace_size()
 * bytes, 256-byte aligned; its contents on entry are ignored.
 * Supported: D in {64, 128}.
 */
int fa_bwd(const void* dout, const void* q, const void* k, const void* v, const void* out, const float* lse,
           void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Sq, int Sk, int H,
           int Hk, int D, float scale, int causal, int window_left, int window_right, const float* alibi_slopes,
           int alibi_batch_stride, int deterministic, fa_stream_t stream);

/* Bytes of device workspace fa_bwd_varlen needs (see fa_bwd_workspace_size). */
size_t fa_bwd_varlen_workspace_size(int B, int total_q, int total_k, int max_seqlen_q, int H, int Hk, int D);

/*
 * Backward over packed sequences: the layouts, cu_seqlens and max_seqlen
 * arguments of fa_fwd_varlen, with dout, q, k, v, out and lse as fa_fwd_varlen
 * takes and writes them. Writes dq (total_q, H, D), dk, dv (total_k, Hk, D)
 * bf16, each sequence's gradients exactly as fa_bwd computes them for that
 * sequence alone. Workspace and precision as fa_bwd.
 */
int fa_bwd_varlen(const void* dout, const void* q, const void* k, const void* v, const void* out, const float* lse,
                  void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int B, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                  int H, int Hk, int D, float scale, int causal, int window_left, int window_right,
                  const float* alibi_slopes, int alibi_batch_stride, int deterministic, fa_stream_t stream);

/*
 * Split count fa_decode_splitkv uses when num_splits == 0, from the SM count of
 * the current device. For the tensor-core split kernel (four or more query
 * pairs per key/value head), while its CTAs per split stay below 0.85 x the SM
 * count: the largest count within that (that many CTAs already draw the whole
 * HBM bandwidth). Otherwise: the fewest splits that fill whole waves.
 */
int fa_decode_num_splits(int B, int Sq, int Sk, int H, int Hk, int D);

/* Bytes of workspace fa_decode_splitkv needs for `num_splits` (0 = auto). */
size_t fa_decode_workspace_size(int B, int Sq, int Sk, int H, int Hk, int D, int num_splits);

/*
 * Split-KV decode for short queries (section "2.2：针对推理进行优化": the
 * key/value loading is split across thread blocks and a separate kernel
 * merges the results). q (B,Sq,H,D) with 1 <= Sq <= 16; k_cache, v_cache
 * (B,Sk,Hk,D) contiguous, Hk dividing H (query head h reads key/value head
 * h / (H / Hk)); a split thread block serves up to four (query row, query
 * head) pairs of one key/value head. Each split writes its normalised partial output and
 * logsumexp to the workspace; the combine kernel merges them exactly,
 * L = log sum_s exp(L_s), O = sum_s exp(L_s - L) O_s, and writes out (bf16)
 * and lse (fp32) in the fa_fwd layouts. Masks and ALiBi as in fa_fwd.
 * num_splits: 0 = auto (fa_decode_num_splits), else 1..256.
 * workspace: >= fa_decode_workspace_size() bytes, 256-byte aligned.
 */
int fa_decode_splitkv(const void* q, const void* k_cache, const void* v_cache, void* out, float* lse,
                      void* workspace, size_t workspace_bytes, int B, int Sq, int Sk, int H, int Hk, int D,
                      float scale, int causal, int window_left, int window_right, const float* alibi_slopes,
                      int alibi_batch_stride, int num_splits, fa_stream_t stream);

/*
 * Split-KV decode over a paged KV cache (section "2.5：分页KV缓存", which only
 * names the feature; the layout here is the reading taken): k_pages, v_pages
 * are (num_pages, page_size, Hk, D) bf16; logical key block p (keys
 * p*page_size .. p*page_size + page_size - 1) of sequence b is page
 * block_table[b * max_pages_per_seq + p]; sequence b has seqlens_k[b] keys.
 * block_table (B, max_pages_per_seq) and seqlens_k (B,) are DEVICE int32
 * arrays, not read back: a length beyond max_pages_per_seq * page_size is
 * clamped to it, and a page index outside [0, num_pages) reads zeros.
 * max_seqlen_k bounds every seqlens_k[b] (it sizes the splits). q, out, lse,
 * masks (anchored at each sequence's own length), ALiBi, num_splits and the
 * workspace (fa_decode_workspace_size with Sk = max_seqlen_k) are those of
 * fa_decode_splitkv. Supported: page_size a multiple of 128, Sq <= 16.
 */
int fa_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                    const int* seqlens_k, void* out, float* lse, void* workspace, size_t workspace_bytes, int B,
                    int Sq, int max_seqlen_k, int num_pages, int page_size, int max_pages_per_seq, int H, int Hk,
                    int D, float scale, int causal, int window_left, int window_right, const float* alibi_slopes,
                    int alibi_batch_stride, int num_splits, fa_stream_t stream);

/*
 * Decode step on a KV cache, appending new keys/values in place and applying
 * rotary embeddings first (section "2.2：针对推理进行优化": flash_attn_with_kvcache
 * "performs rotary embedding and updates the KV cache in place"; the pages give
 * no formula, the standard rotary embedding is the reading taken).
 * Cache: dense k_cache, v_cache (B, cache_rows, Hk, D) when block_table is
 * NULL, else pages (num_pages, page_size, Hk, D) addressed as in
 * fa_decode_paged. cache_seqlens (B,) DEVICE int32: keys already cached.
 * 1. If S_new > 0, rows s of k_new, v_new (B, S_new, Hk, D) are written to
 *    cache position cache_seqlens[b] + s, the keys rotated at that position.
 *    Rows past the cache's capacity (cache_rows, or max_pages_per_seq *
 *    page_size) or on a page index outside [0, num_pages) are not written.
 *    cache_seqlens itself is not updated.
 * 2. Query row i of sequence b is rotated at its diagonal position
 *    i + Sk_b - Sq, Sk_b = min(cache_seqlens[b] + S_new, capacity), and
 *    attends the sequence's Sk_b keys as fa_decode_splitkv does.
 * Rotary (rotary_cos == NULL: none): rotary_cos, rotary_sin (rotary_len,
 * rotary_dim / 2) fp32 on the device; the pair (x1, x2) at frequency f and
 * position t becomes (x1 cos - x2 sin, x1 sin + x2 cos), cos = cos[t][f],
 * pairs (2f, 2f+1) if rotary_interleaved else (f, f + rotary_dim/2); elements
 * at or beyond rotary_dim are unchanged; positions are clamped to
 * [0, rotary_len - 1]. rotary_dim: a multiple of 16, at most D.
 * q, out, lse, masks, ALiBi, num_splits and the workspace
 * (fa_decode_workspace_size with Sk = the capacity) as fa_decode_splitkv.
 */
int fa_decode_kvcache(const void* q, void* k_cache, void* v_cache, const int* cache_seqlens, const void* k_new,
                      const void* v_new, int S_new, const float* rotary_cos, const float* rotary_sin, int rotary_dim,
                      int rotary_len, int rotary_interleaved, const int* block_table, int num_pages, int page_size,
                      int max_pages_per_seq, void* out, float* lse, void* workspace, size_t workspace_bytes, int B,
                      int Sq, int cache_rows, int H, int Hk, int D, float scale, int causal, int window_left,
                      int window_right, const float* alibi_slopes, int alibi_batch_stride, int num_splits,
                      fa_stream_t stream);

/*
 * Split-KV decode that allocates nothing and takes no workspace. The pages
 * have no counterpart to this entry point; it exists for callers that cannot
 * allocate device memory where they run decode (an allocation-free serving
 * loop, a runtime that owns all device memory through its own allocator, a
 * host that forbids allocation after start-up). Arguments, layouts and
 * results are those of fa_decode_splitkv minus the workspace: the split
 * partials live in an 8 MiB array of the library's own device memory, which
 * every GPU that loads the library holds until the process exits.
 * - The array holds only the split partials, B * Sq * H * splits * (D + 1)
 *   fp32 values, each of the two parts rounded up to 256 bytes; it never
 *   holds a rotated query, since this call takes no rotary tables.
 * - num_splits == 0 takes fa_decode_num_splits() and lowers it until the
 *   partials fit in 8 MiB (8388608 bytes). Returns FA_ERR_WORKSPACE if they do
 *   not fit even with one split, or if an explicit num_splits does not fit.
 * - The first call on a device looks up the array's device address (with
 *   that device current); make it before any stream capture.
 * - All calls share the array: calls whose kernels may overlap on the GPU
 *   (other streams, other host threads) race; serialise them. No part of the
 *   array has to start at zero: each call writes every partial it reads.
 */
int fa_decode_splitkv_noalloc(const void* q, const void* k_cache, const void* v_cache, void* out, float* lse,
                              int B, int Sq, int Sk, int H, int Hk, int D, float scale, int causal,
                              int window_left, int window_right, const float* alibi_slopes, int alibi_batch_stride,
                              int num_splits, fa_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the device status word of
 * the current device. Returns FA_OK, FA_ERR_TIMEOUT (a kernel's bounded
 * wait expired; *detail receives the raw word: wait-site code in the low
 * 16 bits) or FA_ERR_CUDA. `detail` may be NULL.
 */
int fa_device_status(fa_stream_t stream, unsigned int* detail);

/* Wait-site code the self-test below records in the device status word. */
#define FA_SELFTEST_SITE 0x7E

/*
 * Diagnostic, outside the method: launches one warp that waits, through the
 * same bounded wait the attention kernels use, on a barrier that nothing
 * arrives at. After about one second the wait gives up and records
 * FA_ERR_TIMEOUT with site FA_SELFTEST_SITE in the device status word, so a
 * following fa_device_status(stream, &d) returns FA_ERR_TIMEOUT with
 * (d & 0xFFFF) == FA_SELFTEST_SITE, and the context stays usable. This lets a
 * caller exercise the failure path on a real GPU without faulting it.
 * Returns FA_OK, or FA_ERR_CUDA if the launch fails.
 */
int fa_selftest_wait_timeout(fa_stream_t stream);

/* Faults fa_debug_set_fault() can inject. */
#define FA_FAULT_NONE 0
#define FA_FAULT_FWD_SKIP_KEY_TILE 1 /* fa_fwd's producer never loads key tile 1 */
#define FA_FAULT_BWD_SKIP_KEY_TILE 2 /* fa_bwd's dQ kernel never loads key tile 1 */

/*
 * Diagnostic, outside the method: exercises the attention kernels' own
 * failure path on a real GPU without faulting it. Sets, for every later
 * launch in this process (all devices), the limit of the kernels' bounded
 * waits (wait_limit_ns; 0 restores the default of one second; otherwise
 * 1 ms .. 1 s) and a fault to inject. With FA_FAULT_FWD_SKIP_KEY_TILE the
 * forward's copy of key tile 1 is left out, so a CTA with at least two key
 * tiles waits for it until the limit, raises its abort flag, lets its copies
 * and tensor-core work in flight finish, frees its tensor memory and returns;
 * fa_device_status() then reports FA_ERR_TIMEOUT with a forward wait site
 * (0x10..0x1F in the low byte of the detail word). FA_FAULT_BWD_SKIP_KEY_TILE
 * does the same in fa_bwd's dQ kernel (sites 0x40..0x4F). The outputs of such
 * a call are undefined. FA_FAULT_NONE with 0 restores normal operation.
 * Returns FA_OK, or FA_ERR_INVALID for an unknown fault or a limit outside
 * that range. Not for use concurrently with normal calls.
 */
int fa_debug_set_fault(int fault, uint64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
