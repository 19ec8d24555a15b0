// Diagnostic for the bounded device-side waits: one CTA waits, with the same helper every TMA/MMA
// pipeline of the library uses, for an mbarrier phase that nothing completes (no arrival, no
// expected copy), so the wait runs out after the given limit.  The expiry is recorded in the
// workspace status word as in the layer kernels, and the kernel then returns normally.
#include "moe_device.cuh"

namespace moe {

__global__ void k_wait_timeout_selftest(int* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    mbar_wait_limit(smem_addr(&bar), 0, reinterpret_cast<volatile int*>(&abort_flag), status,
                    limit_ns);
  __syncthreads();
}

}  // namespace moe

extern "C" moe_status moe_selftest_wait_timeout(void* workspace, int limit_us, moe_stream_t stream) {
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return MOE_ERR_INVALID_ARG;
  if (limit_us < 1 || limit_us > 1000000) return MOE_ERR_INVALID_ARG;
  moe::k_wait_timeout_selftest<<<1, 32, 0, (cudaStream_t)stream>>>(static_cast<int*>(workspace),
                                                                   (uint64_t)limit_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
