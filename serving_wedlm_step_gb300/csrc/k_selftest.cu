// Self-test of the bounded waits: failure detection without a GPU fault.
//
// Every kernel that waits (on a TMA copy, an MMA commit, another warp or
// another block) uses mbar_wait, which gives up after kWaitNs, sets
// WEDLM_DEV_TIMEOUT in the device error word and returns false, so that the
// kernel can drain and return and the CUDA context stays usable.  This
// entry point makes that happen on purpose: one thread waits on a
// shared-memory barrier that nothing ever completes.
#include "internal.h"
#include "tc_ptx.cuh"

namespace wedlm {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(int* word) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival completes it; none is made
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) word[1] = mbar_wait(&bar, 0, word) ? 2 : 1;
}

}  // namespace
}  // namespace wedlm

using namespace wedlm;

extern "C" int wedlm_selftest_bounded_wait(int32_t* word, int32_t* device_error,
                                           int32_t* gave_up, void* stream) {
  if (!word || !device_error || !gave_up || (reinterpret_cast<uintptr_t>(word) & 3))
    return WEDLM_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t host[2] = {0, 0};
  if (cudaMemsetAsync(word, 0, 2 * sizeof(int32_t), st) != cudaSuccess) return WEDLM_ERR_CUDA;
  bounded_wait_selftest_kernel<<<1, 32, 0, st>>>(reinterpret_cast<int*>(word));
  if (cudaGetLastError() != cudaSuccess) return WEDLM_ERR_CUDA;
  if (cudaMemcpyAsync(host, word, sizeof(host), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return WEDLM_ERR_CUDA;
  *device_error = host[0];
  *gave_up = host[1];
  return WEDLM_OK;
}
