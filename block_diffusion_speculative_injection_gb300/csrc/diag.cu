// Diagnostics that exercise the library's failure paths without faulting
// the GPU.
#include "internal.cuh"

namespace dflash {

// One thread waits, with the bounded helper every pipelined kernel uses, on
// an mbarrier that nothing ever arrives on: after the helper's time limit
// it gives up and records a timeout in the context's status word.
__global__ void wait_expires_kernel(int32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  mbar_fence_init();
  mbar_wait(&bar, 0, status);  // phase 0 never completes
}

}  // namespace dflash

using namespace dflash;

extern "C" {

dflash_status dflash_debug_wait_timeout(dflash_ctx* ctx, dflash_stream_t stream) {
  if (!ctx) return DFLASH_E_INVALID_ARG;
  if (launch_k(false, wait_expires_kernel, dim3(1), dim3(32), 0, (cudaStream_t)stream,
               ctx->dev_status) != cudaSuccess)
    return DFLASH_E_CUDA;
  return DFLASH_OK;
}

}  // extern "C"
