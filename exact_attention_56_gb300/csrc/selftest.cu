// Diagnostic kernel: runs the bounded-wait failure path on a real GPU without
// a fault. One warp waits, through the same warp-uniform bounded wait the
// attention kernels use, on an mbarrier that nothing ever arrives at; after
// FA_WAIT_TIMEOUT_NS the wait gives up, raises the CTA abort flag and records
// the timeout with its site code in the device status word, and the kernel
// returns normally, leaving the context usable.
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "internal.h"
#include "ptx.cuh"

namespace fa {

__global__ void __launch_bounds__(32) fa_selftest_wait_kernel(unsigned int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncwarp();
  const Watch w{&abort_flag, status, FA_WAIT_TIMEOUT_NS};
  (void)fa_wait_warp(&bar, 0, w, FA_SELFTEST_SITE);
}

}  // namespace fa

extern "C" int fa_selftest_wait_timeout(fa_stream_t stream) {
  unsigned int* status = fa::device_status_word();
  if (!status) return FA_ERR_CUDA;
  fa::fa_selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
