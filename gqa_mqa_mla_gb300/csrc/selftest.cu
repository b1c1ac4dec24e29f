// selftest.cu -- exercises the bounded mbarrier waits every pipeline uses,
// on the GPU, without a fault: one CTA waits on barriers that nothing ever
// completes, so the waits must give up, set the error flag and let the CTA
// leave.
#include "internal.h"
#include "ptx.cuh"

namespace decattn {
namespace {

// Thread 0 waits on barrier A with a limit of limit_ns and, when it gives up,
// raises the CTA's abort word (as a pipeline role does).  Thread 32 waits on
// barrier B with a limit 1000x longer but watching the abort word, so it must
// leave because of thread 0, long before its own limit.
__global__ void __launch_bounds__(64) wait_timeout_kernel(int* err_flag, int* result,
                                                           uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_word;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    abort_word = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort = &abort_word;
  if (threadIdx.x == 0) {
    const uint64_t t0 = global_timer_ns();
    const bool ok = mbar_wait_or_abort(smem_u32(&bars[0]), 0, err_flag, abort, false, limit_ns);
    result[0] = ok ? 0 : 1;
    result[2] = static_cast<int>((global_timer_ns() - t0) / 1000);  // us waited
  } else if (threadIdx.x == 32) {
    const uint64_t t0 = global_timer_ns();
    const bool ok =
        mbar_wait_or_abort(smem_u32(&bars[1]), 0, err_flag, abort, false, limit_ns * 1000);
    const uint64_t waited = global_timer_ns() - t0;
    result[1] = (!ok && waited < limit_ns * 100) ? 1 : 0;
    result[3] = static_cast<int>(waited / 1000);
  }
  // The plain bounded wait (no abort word) gives up the same way.
  if (threadIdx.x == 1) result[4] = mbar_wait(smem_u32(&bars[0]), 0, err_flag, limit_ns) ? 0 : 1;
}

}  // namespace

cudaError_t launch_wait_selftest(int* err_flag, int* result, uint64_t limit_ns,
                                 cudaStream_t stream) {
  wait_timeout_kernel<<<1, 64, 0, stream>>>(err_flag, result, limit_ns);
  return cudaGetLastError();
}

}  // namespace decattn
