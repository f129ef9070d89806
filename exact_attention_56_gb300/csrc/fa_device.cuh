// Device-side constants shared by the attention kernels: the status word
// layout, the watchdog limit, and the per-row live-key interval.
#pragma once
#include <stdint.h>

namespace fa {

// Device status word: FA_DEV_TIMEOUT is set when a bounded wait gives up;
// the low bits name the wait site (kernel id << 4 | site).
constexpr unsigned int FA_DEV_TIMEOUT = 0x80000000u;
constexpr unsigned int FA_DEV_SITE_MASK = 0x0000FFFFu;
// A legitimate wait inside these kernels lasts microseconds; one second
// means a lost arrival, after which the kernel leaves instead of hanging.
constexpr uint64_t FA_WAIT_TIMEOUT_NS = 1000000000ull;
// Diagnostic fault injection (fa_debug_set_fault), passed to the kernels with
// the wait limit: the forward's producer, or the dQ kernel's, leaves out the
// copy of key tile 1, so the wait for it expires and the kernel takes its
// abort path. Off (0) in every normal call.
constexpr unsigned int FA_INJECT_NONE = 0, FA_INJECT_FWD_SKIP_K = 1, FA_INJECT_BWD_SKIP_K = 2;
// Longest single sleep of a waiting thread before it re-checks the abort flag
// and the watchdog; the thread wakes earlier when the awaited phase completes.
constexpr uint32_t FA_WAIT_SLEEP_NS = 2000u;

// Live key interval of query row i (page "FlashAttention：快速且内存高效的准确注意力机制",
// sections "2.1" and "2.3"): the diagonal key is c(i) = i + Sk - Sq (bottom-right
// alignment); the window keeps keys in [c(i) - left, c(i) + right], -1 meaning
// unbounded, and causal means right = 0. Empty when lo > hi.
struct RowRange {
  int lo, hi;
};

__host__ __device__ __forceinline__ RowRange live_range(int i, int Sq, int Sk, int wl, int wr) {
  const int c = i + Sk - Sq;
  int lo = (wl >= 0) ? c - wl : 0;
  int hi = (wr >= 0) ? c + wr : Sk - 1;
  lo = lo < 0 ? 0 : lo;
  hi = hi > Sk - 1 ? Sk - 1 : hi;
  return RowRange{lo, hi};
}

#ifdef __CUDACC__
// Block coordinates with x as the rank of a CTA's work unit within its (y, z) =
// (head, batch). When the units of one (head, batch) differ in work (masks bounded
// on the right), the grid is renumbered with the rank slowest. The hardware issues
// CTAs roughly in linear order, so each wave then takes the same rank from every
// (head, batch), and the longest units run first across the whole grid, not only
// within one (head, batch). Otherwise consecutive CTAs share a head's K/V in L2,
// which matters more when the units are short.
struct BlockCoord {
  int x, y, z;
};
__device__ __forceinline__ BlockCoord block_coord(bool rank_slowest) {
  if (!rank_slowest) return BlockCoord{int(blockIdx.x), int(blockIdx.y), int(blockIdx.z)};
  const unsigned long long yz = (unsigned long long)gridDim.y * gridDim.z;
  const unsigned long long lin =
      blockIdx.x + (unsigned long long)gridDim.x * (blockIdx.y + (unsigned long long)gridDim.y * blockIdx.z);
  const unsigned int rem = unsigned(lin % yz);
  return BlockCoord{int(lin / yz), int(rem % gridDim.y), int(rem / gridDim.y)};
}
#endif

}  // namespace fa
