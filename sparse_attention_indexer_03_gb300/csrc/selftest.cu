// Self-test of the bounded pipeline wait.  Every mbarrier wait in the
// library's kernels gives up after a cycle budget, or as soon as another warp
// of its CTA raises the CTA's abort flag, and the kernel then reports
// SAI_STATUS_TIMEOUT and drains instead of hanging.  A working pipeline never
// reaches that path, so this launch builds the one situation that does: a
// barrier nothing ever arrives on.  Both ways out are exercised (the budget
// running out; a second warp raising the abort flag after a delay), with the
// same wait primitive the kernels use.
#include "common.cuh"
#include "ptx.cuh"

namespace sai {
namespace {

__global__ void __launch_bounds__(64) bounded_wait_kernel(int mode, long long cycles, uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t b = ptx::smem_addr(&bar);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  if (warp == 0) {
    // Mode 0: the budget is `cycles`.  Mode 1: the budget is the kernels'
    // own (2^31 cycles) and warp 1 raises the abort flag after `cycles`.
    const long long budget = mode == 0 ? cycles : (1LL << 31);
    const bool done = ptx::mbar_wait_warp(b, 0u, reinterpret_cast<volatile int*>(&abort_flag), budget);
    if (!done && lane == 0) raise_status(status, SAI_STATUS_TIMEOUT);
  } else if (mode == 1 && lane == 0) {
    const long long t0 = clock64();
    while (clock64() - t0 < cycles) {
    }
    *reinterpret_cast<volatile int*>(&abort_flag) = 1;
  }
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int mode, long long cycles, uint32_t* status, cudaStream_t stream) {
  bounded_wait_kernel<<<1, 64, 0, stream>>>(mode, cycles, status);
  return cudaGetLastError();
}

}  // namespace sai
