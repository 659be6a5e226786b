// Pieces shared by the tcgen05 kernels (propose_tc.cu, loss_tc.cu): bounded
// mbarrier waits and the driver's tensor-map encoder.
//
// Every mbarrier wait is bounded: after kSpinLimit polls (or the limit the
// caller passes) the waiter records
// DSD_ERR_TIMEOUT, raises the CTA's abort flag (the other roles see it and
// stop issuing work) and returns false.  Nothing traps.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "dsd_common.cuh"
#include "tc_ptx.cuh"

namespace dsd {

constexpr uint32_t kSpinLimit = 1u << 22;        // mbarrier polls before giving up

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         int* status, uint32_t limit = kSpinLimit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort_flag) return false;
  }
  set_status(status, kErrTimeout);
  *abort_flag = 1;
  return false;
}

// The same with acquire at cluster scope, for barriers that the peer CTA of
// a pair arrives on (or whose completions make the peer's writes visible).
__device__ __forceinline__ bool wait_bar_cl(uint64_t* bar, uint32_t parity,
                                            volatile int* abort_flag, int* status) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (tc::mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort_flag) return false;
  }
  set_status(status, kErrTimeout);
  *abort_flag = 1;
  return false;
}
__device__ __forceinline__ bool warp_wait_cl(uint64_t* bar, uint32_t parity,
                                             volatile int* abort_flag, int* status) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_bar_cl(bar, parity, abort_flag, status) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}
__device__ __forceinline__ void drain_bar_cl(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < (1u << 20); ++i)
    if (tc::mbar_try_wait_cluster(bar, parity)) return;
}

// Bounded wait for a counter in global memory that the CTAs of one launch
// (all resident at once) raise: acquire at gpu scope once it reaches target.
// Gives up when the launch's abort word is raised (another CTA failed), or
// after kSpinLimit polls (records DSD_ERR_TIMEOUT and raises the abort word).
__device__ __forceinline__ bool wait_count_gpu(const unsigned int* c, unsigned int target,
                                               unsigned int* abort_word, volatile int* abort_flag,
                                               int* status) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
    if (v >= target) return true;
    if ((i & 31u) == 31u && (*abort_flag || *(volatile unsigned int*)abort_word)) return false;
    __nanosleep(32);
  }
  set_status(status, kErrTimeout);
  atomicExch(abort_word, 1u);
  *abort_flag = 1;
  return false;
}

// Bounded wait that ignores the abort flag: used to drain copies in flight
// before the CTA exits.
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < (1u << 20); ++i)
    if (tc::mbar_try_wait(bar, parity)) return;
}

// Warp-uniform bounded wait: lane 0 polls, the outcome is broadcast, so the
// warp stays converged for the .sync.aligned tcgen05 instructions after it.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int* status, uint32_t limit = kSpinLimit) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, abort_flag, status, limit) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}
__device__ __forceinline__ bool warp_aborted(volatile int* abort_flag) {
  int a = 0;
  if ((threadIdx.x & 31) == 0) a = *abort_flag;
  return __shfl_sync(0xffffffffu, a, 0) != 0;
}

// cuTensorMapEncodeTiled from the driver (nullptr if unavailable); defined in
// propose_tc.cu.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

}  // namespace dsd
