// moe_check_bounded_wait: exercises the bounded wait of the pipelined kernels
// on an mbarrier that nothing completes.  The wait gives up after its limit
// (about one second), the kernel records MOE_DEV_ERR_TIMEOUT and returns: the
// failure path of a stuck pipeline, reached without a fault, a trap or a hang.
#include "moe_common.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_check_kernel(uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    // expects one arrival that never comes
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(&bar))));
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!bounded_wait(&bar, 0u, &abort_flag)) set_status(status, MOE_DEV_ERR_TIMEOUT);
  }
}

}  // namespace
}  // namespace moe

extern "C" int moe_check_bounded_wait(uint32_t* dev_status, moe_stream_t stream) {
  if (!dev_status) return MOE_ERR_INVALID_ARG;
  moe::bounded_wait_check_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(dev_status);
  return moe::counted(cudaGetLastError()) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
