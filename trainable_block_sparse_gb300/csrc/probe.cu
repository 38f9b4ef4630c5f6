// vsa_probe_wait_timeout: exercises the time-out path of the bounded
// mbarrier wait on a barrier that is never completed, so that the recording
// of a device-side time-out and its report through the status word can be
// tested without stalling or faulting the GPU.
#include "../../include/vsa.h"
#include "sm103_ptx.cuh"

namespace vsa {
namespace {

__global__ void probe_wait_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one expected arrival that never comes
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit_ns)) flag_error(status, kDevTimeout);
}

}  // namespace
}  // namespace vsa

extern "C" vsa_status_t vsa_probe_wait_timeout(void* ws, uint32_t limit_us, void* stream) {
  if (!ws || limit_us < 1 || limit_us > 10000000u) return VSA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ws) & 15u) return VSA_ERR_ALIGNMENT;
  vsa::probe_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint32_t*>(ws), static_cast<uint64_t>(limit_us) * 1000ull);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}
