// Self-test of the failure path every kernel of this library relies on: a
// bounded mbarrier wait that nothing completes gives up after its limit,
// records PA_ERR_TIMEOUT in the device status word and lets the kernel
// return, so the context stays usable. Nothing here faults, traps or
// spins without a limit.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

// Wait for the phase with the given parity, giving up after limit_ns of
// global time (same protocol as mbar_wait, with the limit as an argument).
__device__ __forceinline__ bool mbar_wait_limited(uint32_t bar, uint32_t parity, int* status,
                                                  unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) {
      record_error(status, PA_ERR_TIMEOUT);
      return false;
    }
  }
}

// One warp: lane 0 initialises an mbarrier that expects one arrival, which
// never comes, and waits for its first phase.
__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(unsigned long long limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait_limited(smem_u32(&bar), 0, status, limit_ns);
  __syncwarp();
}

}  // namespace pa

using namespace pa;

extern "C" {

int pa_selftest_bounded_wait(int64_t limit_ns, void* stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000LL) return PA_ERR_ARG;
  int* st = device_status_ptr();
  if (!st) return PA_ERR_CUDA;
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((unsigned long long)limit_ns, st);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"
