// Hardware-aware batch-global prefix scheduler ("DSpark 论文精读：置信度调度推测
// 解码、半自回归生成与大模型推理加速", section 3.2).
//
// One CTA of 1024 threads:
//   1. key every (r, j) slot by survival descending, then r, then j:
//      key = ~ord(a) << 32 | (r * gamma + j)  (ascending key order);
//   2. bitonic sort of the keys in shared memory (R * gamma <= 4096);
//   3. inclusive fp64 scan of the sorted survivals; tau_k = R + prefix_k,
//      Theta_k = tau_k * SPS(R + k) for the feasible cuts k = 1..min(Rg, n_sps - R),
//      Theta_0 = R * SPS(R);
//   4. argmax over k (largest Theta, smallest k on ties);
//   5. keep_len[r] = number of the first k* sorted slots that belong to r.
// fp64 running sums of fp32 survivals are exact whenever the survivals span
// less than ~2^18 in magnitude, so the cut is the same as an exact one.
#include "dsd_common.cuh"

namespace dsd {

constexpr int kSchedThreads = 1024;

struct SchedParams {
  const float* survival;
  const float* sps;
  int32_t* keep_len;
  float* theta_B;
  int* status;
  int R, gamma, n_sps, NP;
};

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(SchedParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem);
  int* cnt = reinterpret_cast<int*>(smem + (size_t)p.NP * sizeof(unsigned long long));
  __shared__ double warp_tot[32];
  __shared__ double warp_best_t[32];
  __shared__ int warp_best_k[32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = p.R * p.gamma;
  const int NP = p.NP;

  for (int i = tid; i < NP; i += kSchedThreads) {
    unsigned long long k = ~0ull;
    if (i < N) {
      float a = p.survival[i];
      if (!isfinite(a)) {
        set_status(p.status, kErrNonfinite);
        a = 0.f;
      }
      k = ((unsigned long long)(~f2ord(a)) << 32) | (unsigned long long)i;
    }
    keys[i] = k;
  }
  for (int r = tid; r < p.R; r += kSchedThreads) cnt[r] = 0;
  __syncthreads();

  // bitonic sort, ascending
  for (int k = 2; k <= NP; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < NP; i += kSchedThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long x = keys[i], y = keys[ixj];
          const bool up = (i & k) == 0;
          if ((x > y) == up) {
            keys[i] = y;
            keys[ixj] = x;
          }
        }
      }
      __syncthreads();
    }
  }

  // each thread owns IPT consecutive sorted items
  const int IPT = (NP + kSchedThreads - 1) / kSchedThreads;
  const int i0 = tid * IPT;
  double local = 0.0;
  for (int t = 0; t < IPT; ++t) {
    const int i = i0 + t;
    if (i < N) local += (double)ord2f(~(uint32_t)(keys[i] >> 32));
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
    double w = warp_tot[lane];
    double wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
  }
  __syncthreads();
  double run = warp_tot[warp] + (incl - local);

  const int Kmax = min(N, p.n_sps - p.R);
  double best_t = -INFINITY;
  int best_k = 0x7fffffff;
  for (int t = 0; t < IPT; ++t) {
    const int i = i0 + t;
    if (i < N) run += (double)ord2f(~(uint32_t)(keys[i] >> 32));
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
    best_t = warp_best_t[lane];
    best_k = warp_best_k[lane];
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
  for (int i = tid; i < kstar; i += kSchedThreads) {
    const int item = (int)(keys[i] & 0xFFFFFFFFull);
    atomicAdd(&cnt[item / p.gamma], 1);
  }
  __syncthreads();
  for (int r = tid; r < p.R; r += kSchedThreads) p.keep_len[r] = cnt[r];
  if (tid == 0 && p.theta_B) {
    p.theta_B[0] = (float)warp_best_t[0];
    p.theta_B[1] = (float)(p.R + kstar);
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
  p.R = R;
  p.gamma = ctx.cfg.gamma;
  p.n_sps = n_sps;
  int NP = 2;
  while (NP < R * ctx.cfg.gamma) NP <<= 1;
  p.NP = NP;
  const size_t smem = (size_t)NP * sizeof(unsigned long long) + (size_t)R * sizeof(int);
  cudaError_t e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  schedule_kernel<<<1, kSchedThreads, smem, s>>>(p);
  count_launch(ctx);
  return cudaGetLastError();
}

}  // namespace dsd
