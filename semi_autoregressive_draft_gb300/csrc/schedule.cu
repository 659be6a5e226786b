// Hardware-aware batch-global prefix scheduler ("DSpark 论文精读：置信度调度推测
// 解码、半自回归生成与大模型推理加速", section 3.2).
//
// The scheduler's order is survival descending, then request, then position,
// i.e. slot index i = r * gamma + j ascending on ties.  One launch over many
// SMs:
//   1. rank: every CTA stages all survivals in shared memory; one warp per
//      slot counts the slots that precede it in that order (an O(N^2) count
//      spread over the grid, N = R * gamma <= 4096), which is its position,
//      and writes order[position] = slot.  Ranks form a permutation because
//      the order is total.
//   2. the last CTA to finish (a ticket counter, reset by that CTA) takes
//      the sorted slots: inclusive fp64 scan of the survivals in that order;
//      tau_k = R + prefix_k, Theta_k = tau_k * SPS(R + k) for the feasible cuts
//      k = 1..min(N, n_sps - R), Theta_0 = R * SPS(R); argmax over k (largest
//      Theta, smallest k on ties); keep_len[r] = number of the first k* sorted
//      slots that belong to r.
// fp64 running sums of fp32 survivals are exact whenever the survivals span
// less than ~2^18 in magnitude, so the cut is the same as an exact one.
#include "dsd_common.cuh"

namespace dsd {

constexpr int kSchedThreads = 256;
constexpr int kSchedWarps = kSchedThreads / 32;

struct SchedParams {
  const float* survival;
  const float* sps;
  int32_t* keep_len;
  float* theta_B;
  int* status;
  int* order;              // [N] slot at each sorted position
  unsigned int* ticket;    // zero between calls
  int R, gamma, n_sps;
};

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(SchedParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int N = p.R * p.gamma;
  float* s_a = reinterpret_cast<float*>(smem);                 // [N] survivals
  int* cnt = reinterpret_cast<int*>(smem + (size_t)N * sizeof(float));   // [R]
  __shared__ double warp_tot[kSchedWarps];
  __shared__ double warp_best_t[kSchedWarps];
  __shared__ int warp_best_k[kSchedWarps];
  __shared__ int am_last;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int i = tid; i < N; i += kSchedThreads) {
    float a = p.survival[i];
    if (!isfinite(a)) {
      if (blockIdx.x == 0) set_status(p.status, kErrNonfinite);
      a = 0.f;
    }
    s_a[i] = a;
  }
  __syncthreads();

  // ---- 1. rank of each slot in the schedule order ----
  for (int i = blockIdx.x * kSchedWarps + warp; i < N; i += gridDim.x * kSchedWarps) {
    const float ai = s_a[i];
    int c = 0;
    for (int i2 = lane; i2 < N; i2 += 32) {
      const float a2 = s_a[i2];
      c += (a2 > ai || (a2 == ai && i2 < i)) ? 1 : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) p.order[c] = i;
  }

  // ---- the last CTA to arrive finishes the schedule ----
  __threadfence();
  __syncthreads();
  if (tid == 0) am_last = (atomicAdd(p.ticket, 1u) == gridDim.x - 1) ? 1 : 0;
  __syncthreads();
  if (!am_last) return;
  __threadfence();
  for (int r = tid; r < p.R; r += kSchedThreads) cnt[r] = 0;

  // ---- 2. prefix sums in schedule order, Theta, argmax, allocation ----
  // each thread owns IPT consecutive sorted positions
  const int IPT = (N + kSchedThreads - 1) / kSchedThreads;
  const int i0 = tid * IPT;
  double local = 0.0;
  for (int t = 0; t < IPT; ++t) {
    const int i = i0 + t;
    if (i < N) local += (double)s_a[__ldcg(&p.order[i])];
  }
  // exclusive block scan of the per-thread sums
  double incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const double w = lane < kSchedWarps ? warp_tot[lane] : 0.0;
    double wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < kSchedWarps) warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
  }
  __syncthreads();
  double run = warp_tot[warp] + (incl - local);

  const int Kmax = min(N, p.n_sps - p.R);
  double best_t = -INFINITY;
  int best_k = 0x7fffffff;
  for (int t = 0; t < IPT; ++t) {
    const int i = i0 + t;
    if (i < N) run += (double)s_a[__ldcg(&p.order[i])];
    const int k = i + 1;
    if (k <= Kmax) {
      const double theta = ((double)p.R + run) * (double)p.sps[p.R + k - 1];
      if (theta > best_t) {
        best_t = theta;
        best_k = k;
      }
    }
  }
  // argmax: larger Theta, then smaller k
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double ot = __shfl_xor_sync(0xffffffffu, best_t, o);
    const int ok = __shfl_xor_sync(0xffffffffu, best_k, o);
    if (ot > best_t || (ot == best_t && ok < best_k)) {
      best_t = ot;
      best_k = ok;
    }
  }
  if (lane == 0) {
    warp_best_t[warp] = best_t;
    warp_best_k[warp] = best_k;
  }
  __syncthreads();
  if (warp == 0) {
    best_t = lane < kSchedWarps ? warp_best_t[lane] : -INFINITY;
    best_k = lane < kSchedWarps ? warp_best_k[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double ot = __shfl_xor_sync(0xffffffffu, best_t, o);
      const int ok = __shfl_xor_sync(0xffffffffu, best_k, o);
      if (ot > best_t || (ot == best_t && ok < best_k)) {
        best_t = ot;
        best_k = ok;
      }
    }
    if (lane == 0) {
      const double theta0 = (double)p.R * (double)p.sps[p.R - 1];
      if (!(best_t > theta0)) {
        best_t = theta0;
        best_k = 0;
      }
      warp_best_t[0] = best_t;
      warp_best_k[0] = best_k;
    }
  }
  __syncthreads();
  const int kstar = warp_best_k[0];
  for (int i = tid; i < kstar; i += kSchedThreads) atomicAdd(&cnt[__ldcg(&p.order[i]) / p.gamma], 1);
  __syncthreads();
  for (int r = tid; r < p.R; r += kSchedThreads) p.keep_len[r] = cnt[r];
  if (tid == 0) {
    if (p.theta_B) {
      p.theta_B[0] = (float)warp_best_t[0];
      p.theta_B[1] = (float)(p.R + kstar);
    }
    *p.ticket = 0u;   // ready for the next call (kernels on the stream run in order)
  }
}

cudaError_t launch_schedule(const Ctx& ctx, int R, const float* survival, const float* sps,
                            int n_sps, int32_t* keep_len, float* theta_B, cudaStream_t s) {
  SchedParams p{};
  p.survival = survival;
  p.sps = sps;
  p.keep_len = keep_len;
  p.theta_B = theta_B;
  p.status = ctx.ws.status;
  p.order = ctx.ws.sched_order;
  p.ticket = ctx.ws.tickets + 0;
  p.R = R;
  p.gamma = ctx.cfg.gamma;
  p.n_sps = n_sps;
  const int N = R * ctx.cfg.gamma;
  // one warp per slot, at most one CTA per SM
  int grid = (N + kSchedWarps - 1) / kSchedWarps;
  if (grid > ctx.num_sms) grid = ctx.num_sms;
  const size_t smem = (size_t)N * sizeof(float) + (size_t)R * sizeof(int);
  schedule_kernel<<<grid, kSchedThreads, smem, s>>>(p);
  count_launch(ctx);
  return cudaGetLastError();
}

}  // namespace dsd
