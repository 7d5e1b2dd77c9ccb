// Self-test of the bounded waits: every wait in this library's kernels (an
// mbarrier phase, a device flag) gives up after a limit of device wall time,
// records PA_DEVERR_TIMEOUT and lets the kernel return, so that a wait that
// can never be satisfied leaves the context usable instead of hanging it.
// This kernel makes two such waits run out on purpose: an mbarrier phase
// that no thread or copy completes, and a device word that no code writes.
#include "pa_internal.h"
#include "ptx.cuh"

namespace pa {
namespace {

__device__ int32_t g_never_set;  // zero-initialised; nothing writes it

__global__ void bounded_wait_selftest_kernel(int32_t* err, uint64_t limit_ns, uint64_t* elapsed) {
  __shared__ __align__(8) uint64_t s_bar;
  const uint32_t bar = smem_addr(&s_bar);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);  // phase 0 completes on one arrival, and none comes
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t t0 = global_timer_ns();
  const bool got_bar = mbar_wait_bounded(bar, 0, limit_ns);
  const uint64_t t1 = global_timer_ns();
  bool got_flag = ld_acquire_gpu(&g_never_set) != 0;
  while (!got_flag && global_timer_ns() - t1 <= limit_ns) got_flag = ld_acquire_gpu(&g_never_set) != 0;
  const uint64_t t2 = global_timer_ns();
  if (threadIdx.x == 0) {
    if (!got_bar || !got_flag) atomicOr(err, PA_DEVERR_TIMEOUT);
    if (elapsed) {
      elapsed[0] = t1 - t0;
      elapsed[1] = t2 - t1;
    }
  }
}

}  // namespace

cudaError_t bounded_wait_selftest(int32_t* err, uint64_t limit_ns, uint64_t* elapsed,
                                  cudaStream_t s) {
  bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(err, limit_ns, elapsed);
  return cudaGetLastError();
}

}  // namespace pa
