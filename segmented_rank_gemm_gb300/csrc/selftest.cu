// selftest.cu -- a self-test of the bounded waits every pipeline kernel of this library uses.
//
// A wait that never completes (a flag nothing sets, an mbarrier phase nobody arrives on)
// must give up after its bound, raise the timeout flag and return, leaving the context
// usable -- it must not hang the GPU.  lora_wait_selftest runs exactly such a wait.
#include <cuda_runtime.h>

#include "lora_common.cuh"
#include "lora_layer.h"

namespace lora {

// which = 0: wait for a global flag nothing sets (the stream-K hand-over wait);
// which = 1: wait for an mbarrier phase nobody arrives on (the pipeline waits).
// flag_err[0] is the flag (0), flag_err[1] receives the error flags.
__global__ void wait_selftest_kernel(int which, int32_t* flag_err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  if (which == 0) {
    wait_flag_gpu(flag_err, 1, flag_err + 1);
  } else {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_wait(&bar, 0u, flag_err + 1);  // phase 0 completes only on an arrival
  }
}

}  // namespace lora

extern "C" int lora_wait_selftest(int which, void* stream_) {
  if (which != 0 && which != 1) return LORA_EINVAL;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int32_t* buf = nullptr;
  if (cudaMalloc(&buf, 2 * sizeof(int32_t)) != cudaSuccess) {
    cudaGetLastError();
    return LORA_ENOMEM;
  }
  int32_t host[2] = {0, 0};
  int rc = LORA_ECUDA;
  if (cudaMemsetAsync(buf, 0, 2 * sizeof(int32_t), stream) == cudaSuccess) {
    lora::wait_selftest_kernel<<<1, 32, 0, stream>>>(which, buf);
    if (cudaGetLastError() == cudaSuccess &&
        cudaMemcpyAsync(host, buf, sizeof(host), cudaMemcpyDeviceToHost, stream) == cudaSuccess &&
        cudaStreamSynchronize(stream) == cudaSuccess)
      rc = (host[1] & LORA_ERRF_TIMEOUT) ? LORA_ETIMEOUT : LORA_OK;
  }
  cudaFree(buf);
  return rc;
}
