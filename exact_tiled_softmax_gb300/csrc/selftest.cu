// Self-test of the bounded-wait path that every tensor-core kernel uses: a
// wait on an mbarrier that nothing ever arrives on must give up after its
// limit, record EXATTN_TIMEOUT in the status word and let the kernel return;
// a second waiter must notice the abort flag and return as well.
#include "common.cuh"
#include "tc_ptx.cuh"
#include "../../include/exattn.h"

namespace exattn {
namespace {

using namespace tc;

__global__ void __launch_bounds__(64, 1)
    selftest_wait_kernel(unsigned* status, unsigned long long limit_ns, unsigned* result) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort = &abort_flag;
  if (lane == 0) {
    const uint64_t t0 = globaltimer_ns();
    if (warp == 0) {
      // Nothing arrives on bars[0]: this wait must run out after limit_ns.
      if (!mbar_wait(smem_u32(&bars[0]), 0, abort, limit_ns)) {
        raise_status(status, kStatusTimeout);
        *abort = 1;
        result[0] = 1u;
      }
    } else {
      // Nothing arrives on bars[1] either, but this waiter has the default
      // limit: it must stop because of the abort flag, long before that.
      const bool ok = mbar_wait(smem_u32(&bars[1]), 0, abort);
      result[1] = ok ? 0u : 1u;
      result[2] = static_cast<unsigned>((globaltimer_ns() - t0) / 1000u);  // microseconds
    }
  }
  __syncthreads();
}

}  // namespace
}  // namespace exattn

extern "C" int exattn_selftest_wait_timeout(void* workspace, unsigned limit_us, void* cuda_stream) {
  if (!workspace || limit_us == 0 || limit_us > 100000) return EXATTN_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return EXATTN_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  unsigned* status = static_cast<unsigned*>(workspace);
  if (cudaMemsetAsync(workspace, 0, 256, s) != cudaSuccess) return EXATTN_CUDA_ERROR;
  exattn::selftest_wait_kernel<<<1, 64, 0, s>>>(status, 1000ull * limit_us, status + 1);
  return cudaGetLastError() == cudaSuccess ? EXATTN_OK : EXATTN_CUDA_ERROR;
}
