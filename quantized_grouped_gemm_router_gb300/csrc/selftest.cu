// Failure-detection self-test of the bounded waits (no GPU fault, trap or hang): one thread waits
// on an mbarrier that nothing arrives on, through the same bounded wait the prefill GEMM and decode
// kernels use; the wait gives up after kWaitCycles, the thread records MOE_ERR_DEVICE_TIMEOUT in the
// workspace's sticky status word, and the kernel returns, leaving the context usable.
#include <cuda_runtime.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(WsHeader* hdr) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);  // expects one arrival, which never comes
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && !mbar_wait(b, 0, &abort_flag)) set_device_status(hdr, MOE_ERR_DEVICE_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(WsHeader* hdr, cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>(hdr);
  return cudaGetLastError();
}

}  // namespace moe
