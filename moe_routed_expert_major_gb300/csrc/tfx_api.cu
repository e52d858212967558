// tfx_api.cu -- error strings, version, and the bounded-wait self-test.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tfx_common.cuh"

namespace tfx {

// One block waits on an mbarrier that nothing will complete: the bounded wait must run out,
// report TFX_ST_TIMEOUT and return.
__global__ void wait_timeout_kernel(int32_t* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0u, timeout_ns)) report(status, TFX_ST_TIMEOUT);
  __syncthreads();
  if (threadIdx.x == 0) mbar_arrive(&bar);  // complete the phase before the block exits
  __syncthreads();
}

}  // namespace tfx

extern "C" const char* tfx_strerror(int code) {
  switch (code) {
    case TFX_OK: return "ok";
    case TFX_EINVAL: return "invalid argument (null or misaligned pointer, bad sizes)";
    case TFX_EUNSUPPORTED: return "unsupported shape for these kernels";
    case TFX_ELAUNCH: return "CUDA launch failed";
    case TFX_ECUDA: return "CUDA device query failed";
    default: return "unknown error";
  }
}

extern "C" int tfx_version(void) { return 1; }

extern "C" int tfx_selftest_wait_timeout(int32_t* status, int64_t timeout_ns, void* stream) {
  if (!status || timeout_ns <= 0 || timeout_ns > 10000000000ll) return TFX_EINVAL;
  tfx::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, (uint64_t)timeout_ns);
  return cudaGetLastError() == cudaSuccess ? TFX_OK : TFX_ELAUNCH;
}
