// Self-test of the bounded mbarrier waits that every tensor-core kernel of
// the library relies on (tc_common.cuh): one CTA whose barriers are never
// completed, so that the waits run out exactly as they would if a copy or a
// peer role never arrived.  No copy, no tensor-core operation and no other
// CTA is involved, so nothing is left in flight when the kernel returns.
//
//   warp 0  initialises barrier X with two expected arrivals and barrier Y
//           with one, then arrives on X once: neither phase 0 can complete;
//   warp 1  waits on X with the caller's short poll limit: the wait gives up,
//           records DSD_ERR_TIMEOUT in the status word and raises the CTA's
//           abort flag (what a timed-out role does in the real kernels);
//   warp 2  waits on Y with the full limit: it sees the abort flag within 256
//           polls of its raising and stops waiting without a status of its
//           own (what the other roles of a real kernel do).
// roles_out[0] / [1] receive 1 if warp 1 / warp 2 returned from its wait
// with the phase complete (expected: 0 and 0), roles_out[2] the number of
// warps that left their wait (expected: 2).
#include "tc_common.cuh"

namespace dsd {

namespace {

__global__ void __launch_bounds__(96, 1)
    wait_selftest_kernel(uint32_t poll_limit, int* status, int32_t* roles_out) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  __shared__ int left;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bars[0], 2);
    tc::mbar_init(&bars[1], 1);
    abort_flag = 0;
    left = 0;
    tc::mbar_fence_init();
  }
  __syncthreads();
  volatile int* ab = &abort_flag;
  if (warp == 0) {
    if (lane == 0) tc::mbar_arrive(&bars[0]);   // one of the two arrivals X expects
  } else {
    const bool ok = warp == 1 ? warp_wait(&bars[0], 0, ab, status, poll_limit)
                              : warp_wait(&bars[1], 0, ab, status);
    if (lane == 0) {
      atomicAdd(&left, 1);
      if (roles_out) roles_out[warp - 1] = ok ? 1 : 0;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && roles_out) roles_out[2] = left;
}

}  // namespace

cudaError_t launch_wait_selftest(const Ctx& ctx, uint32_t poll_limit, int32_t* roles_out,
                                 cudaStream_t s) {
  wait_selftest_kernel<<<1, 96, 0, s>>>(poll_limit, ctx.ws.status, roles_out);
  count_launch(ctx);
  return cudaGetLastError();
}

}  // namespace dsd
