// Check of the bounded-wait path every pipelined kernel relies on (sm_103a).
//
// The kernels that wait on mbarriers (the scoring pipeline, the tcgen05 latent
// attention) give up after a clock64 limit, set SKV_DEV_TIMEOUT in the caller's
// status word and return, so a lost arrival never hangs the GPU.  This kernel runs
// the same helper, wait_or_abort, on a barrier that nothing completes (arrive == 0)
// or that one thread completes first (arrive == 1), with a caller-chosen limit: the
// first case must end with SKV_DEV_TIMEOUT set, the second with nothing set.
#include "skv_internal.cuh"

namespace skv {
namespace {

__global__ void __launch_bounds__(64) wait_check_kernel(long long limit_cycles, int arrive, int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int s_abort;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    s_abort = 0;
  }
  __syncthreads();
  if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
  wait_or_abort(&bar, 0u, &s_abort, status, limit_cycles);
}

}  // namespace

skv_status launch_wait_check(long long limit_cycles, int arrive, int32_t* status, cudaStream_t st) {
  wait_check_kernel<<<1, 64, 0, st>>>(limit_cycles, arrive, status);
  SKV_LAUNCH_CHECK();
  return SKV_OK;
}

}  // namespace skv
