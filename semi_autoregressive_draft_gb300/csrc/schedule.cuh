// Hardware-aware batch-global prefix scheduler ("DSpark 论文精读：置信度调度推测
// 解码、半自回归生成与大模型推理加速", section 3.2): device code shared by the
// standalone schedule kernel and the proposal's finalize kernel, which runs
// the schedule in extra CTAs when a whole cycle is launched at once.
//
// The scheduler's order is survival descending, then request, then position,
// i.e. slot index i = r * gamma + j ascending on ties.  Each slot becomes the
// 64-bit key ord(a) << 32 | ~i, unique and larger for earlier slots, so the
// order is the keys' descending order.  Cut k keeps the first k slots of the
// order: tau_k = R + prefix_k, Theta_k = tau_k * SPS(R + k), Theta_0 =
// R * SPS(R); the allocation is the cut with the largest Theta (the smallest
// k on ties) among the feasible ones, k <= min(N, n_sps - R).
//
// Slot x sits at position c_x = #{keys above x} of the order, and the cut
// that ends with it, k = c_x + 1, has prefix_k = sum of the survivals of the
// keys at or above x.  Both are sums over all slots, so no sort is needed:
//   1. every CTA stages all keys and survivals in shared memory (survivals
//      clamped to [0, 1], as integers in units of 2^-48: each rounds by at
//      most 2^-49 and the sum of 4096 stays below 2^61, so every prefix is
//      exact and independent of the order of the additions);
//   2. one warp per slot counts and sums over all slots; lane 0 forms
//      Theta_k in fp64, writes its order-preserving bit pattern to
//      theta_bits[c_x] and the slot to order[c_x], and raises the grid-wide
//      maximum with an integer atomicMax (a non-negative fp64 compares like
//      its bits, so the maximum is exact without fp64 comparisons);
//   3. the last CTA to finish (a ticket) compares the maximum with Theta_0,
//      takes the smallest k whose Theta has the maximum's bits, counts the
//      kept slots per request and resets the maximum and the ticket.
#pragma once
#include "dsd_common.cuh"

namespace dsd {

constexpr int kSchedThreads = 256;
constexpr int kSchedWarps = kSchedThreads / 32;
constexpr float kFixScaleF = 281474976710656.0f;          // 2^48
constexpr double kInvFixScale = 1.0 / 281474976710656.0;

struct SchedParams {
  const float* survival;            // [R, gamma], or nullptr: survivals from conf
  const float* conf;                // [R, gamma] confidences (when survival is nullptr)
  const float* sps;
  int32_t* keep_len;
  float* theta_B;
  int* status;
  unsigned long long* theta_bits;   // [N] order-preserving bits of Theta at each cut
  int* order;                       // [N] slot at each position of the order
  unsigned long long* best;         // grid-wide maximum of theta_bits; zero between calls
  unsigned int* ticket;             // zero between calls
  int R, gamma, n_sps;
};

// Order-preserving map of an fp64 value to 64 bits (larger value, larger bits).
__device__ __forceinline__ unsigned long long d2ord(double d) {
  const unsigned long long u = (unsigned long long)__double_as_longlong(d);
  return (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
}
__device__ __forceinline__ double ord2d(unsigned long long o) {
  const unsigned long long u = (o & 0x8000000000000000ull) ? (o ^ 0x8000000000000000ull) : ~o;
  return __longlong_as_double((long long)u);
}

// One CTA's share of the schedule: CTA `cta` of `n_ctas` (all of them run
// this with kSchedThreads threads and schedule_smem_bytes of dynamic shared
// memory).
__device__ __forceinline__ void schedule_cta(const SchedParams& p, int cta, int n_ctas,
                                             unsigned char* smem) {
  const int N = p.R * p.gamma;
  unsigned long long* s_key = reinterpret_cast<unsigned long long*>(smem);   // [N]
  long long* s_fx = reinterpret_cast<long long*>(s_key + N);                 // [N]
  int* cnt = reinterpret_cast<int*>(s_fx + N);                               // [R] (last CTA), then 2 flags

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int& am_last = *reinterpret_cast<int*>(cnt + p.R);
  int& s_kmin = *(reinterpret_cast<int*>(cnt + p.R) + 1);

  // ---- 1. keys and fixed-point survivals ----
  if (p.survival) {
    for (int i = tid; i < N; i += kSchedThreads) {
      float a = p.survival[i];
      if (!isfinite(a)) {
        if (cta == 0) set_status(p.status, kErrNonfinite);
        a = 0.f;
      }
      a = fminf(fmaxf(a, 0.f), 1.f) + 0.f;   // + 0 turns -0 into +0
      s_key[i] = make_key(a, (uint32_t)i);
      s_fx[i] = __float2ll_rn(a * kFixScaleF);   // exact scaling by 2^48
    }
  } else {
    // survivals straight from the confidences, computed exactly as the
    // proposal's finalize computes its survival output (fp64 product of the
    // clamped confidences, rounded to fp32); non-finite ones are reported
    // there
    for (int r = tid; r < p.R; r += kSchedThreads) {
      double acc = 1.0;
      for (int j = 0; j < p.gamma; ++j) {
        const int i = r * p.gamma + j;
        float c = p.conf[i];
        c = isfinite(c) ? fminf(fmaxf(c, 0.f), 1.f) : 0.f;
        acc *= (double)c;
        const float a = (float)acc + 0.f;
        s_key[i] = make_key(a, (uint32_t)i);
        s_fx[i] = __float2ll_rn(a * kFixScaleF);
      }
    }
  }
  __syncthreads();

  // ---- 2. position and prefix of every slot; Theta at its cut ----
  const int Kmax = min(N, p.n_sps - p.R);
  for (int x = cta * kSchedWarps + warp; x < N; x += n_ctas * kSchedWarps) {
    const unsigned long long kx = s_key[x];
    int c = 0;
    long long pre = 0;
#pragma unroll 4
    for (int y = lane; y < N; y += 32) {
      const unsigned long long ky = s_key[y];
      const long long fy = s_fx[y];
      c += ky > kx ? 1 : 0;
      pre += ky >= kx ? fy : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      c += __shfl_xor_sync(0xffffffffu, c, o);
      pre += __shfl_xor_sync(0xffffffffu, pre, o);
    }
    if (lane == 0) {
      unsigned long long bits = 0ull;   // below every value: not a candidate
      if (c < Kmax) {                   // cut k = c + 1 is feasible
        const long long tau = (long long)p.R * (1ll << 48) + pre;
        const double theta = ((double)tau * kInvFixScale) * (double)__ldg(&p.sps[p.R + c]);
        if (theta == theta) {           // a NaN Theta never wins
          bits = d2ord(theta);
          atomicMax(p.best, bits);
        }
      }
      p.theta_bits[c] = bits;
      p.order[c] = x;
    }
  }

  // ---- 3. the last CTA to arrive finishes the schedule ----
  __threadfence();
  __syncthreads();
  if (tid == 0) am_last = (atomicAdd(p.ticket, 1u) == (unsigned int)n_ctas - 1u) ? 1 : 0;
  __syncthreads();
  if (!am_last) return;
  __threadfence();
  const unsigned long long best = __ldcg(p.best);
  const double theta0 = (double)p.R * (double)__ldg(&p.sps[p.R - 1]);
  // Theta_0 wins unless a cut is strictly larger (a NaN Theta_0 also stays)
  const bool cut = best != 0ull && !(theta0 != theta0) && best > d2ord(theta0);
  if (tid == 0) s_kmin = 0x7fffffff;
  for (int r = tid; r < p.R; r += kSchedThreads) cnt[r] = 0;
  __syncthreads();
  if (cut)
    for (int c = tid; c < N; c += kSchedThreads)
      if (__ldcg(&p.theta_bits[c]) == best) atomicMin(&s_kmin, c + 1);
  __syncthreads();
  const int kstar = cut ? s_kmin : 0;
  for (int c = tid; c < kstar; c += kSchedThreads)
    atomicAdd(&cnt[__ldcg(&p.order[c]) / p.gamma], 1);
  __syncthreads();
  for (int r = tid; r < p.R; r += kSchedThreads) p.keep_len[r] = cnt[r];
  if (tid == 0) {
    if (p.theta_B) {
      p.theta_B[0] = (float)(cut ? ord2d(best) : theta0);
      p.theta_B[1] = (float)(p.R + kstar);
    }
    *p.best = 0ull;     // ready for the next call (kernels on the stream run in order)
    *p.ticket = 0u;
  }
}


// Dynamic shared memory of a schedule CTA: keys and fixed-point survivals of
// the N = R * gamma slots, the per-request counts and two flags.
inline size_t schedule_smem_bytes(int R, int gamma) {
  return (size_t)R * gamma * 16 + (size_t)R * sizeof(int) + 2 * sizeof(int);
}

// Host side, in schedule.cu: the parameters of a schedule over the context's
// workspace, and the number of CTAs it runs on.
SchedParams make_sched_params(const Ctx& ctx, int R, const float* survival, const float* conf,
                              const float* sps, int n_sps, int32_t* keep_len, float* theta_B);
int schedule_ctas(const Ctx& ctx, int R);

}  // namespace dsd
