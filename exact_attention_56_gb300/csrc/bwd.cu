// Backward attention kernels (placeholder until the tcgen05 backward lands).
#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "internal.h"

namespace fa {

size_t bwd_workspace_bytes(int B, int Sq, int Sk, int H, int D, int deterministic) {
  (void)Sk;
  (void)deterministic;
  return size_t(B) * Sq * H * D * 4 + size_t(B) * H * Sq * 4 + 512;
}

int bwd_launch(const AttnShape&, const void*, const void*, const void*, const void*, const void*, const float*,
               void*, void*, void*, void*, int, cudaStream_t) {
  return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
