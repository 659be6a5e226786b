// Offline teacher-forced overlap metrics ("Qwen3.8-Flash-Next DSpark 训练实验",
// 评估口径 / 离线指标; "DSpark 论文精读" 3.1 overlap identity).
//
// overlap_rows: one CTA per (block n, position i).  Invalid positions write
// zeros and return.  Pass 1 streams the P and Q rows once (16-byte loads)
// into base-2 online log-sum-exp states; pass 2 re-reads them (hitting L2:
// the CTAs in flight hold a few tens of MB) and accumulates
// sum min(p, q) and sum |p - q| with p, q formed from the two normalisers.
// overlap_finalize: one CTA; tau per block, accept_rate per position over
// the valid blocks, mean tau over the valid blocks, all summed in a fixed
// order in fp64 so the result does not depend on scheduling.
#include "dsd_common.cuh"

namespace dsd {

constexpr int kOvThreads = 512;

template <typename T>
__device__ __forceinline__ int load_chunk(const T* row, int v0, float* x) {
  const uint4 q = ld_stream16(row + v0);
  if constexpr (sizeof(T) == 2) {
    x[0] = bf16lo(q.x); x[1] = bf16hi(q.x); x[2] = bf16lo(q.y); x[3] = bf16hi(q.y);
    x[4] = bf16lo(q.z); x[5] = bf16hi(q.z); x[6] = bf16lo(q.w); x[7] = bf16hi(q.w);
    return 8;
  } else {
    x[0] = __uint_as_float(q.x); x[1] = __uint_as_float(q.y);
    x[2] = __uint_as_float(q.z); x[3] = __uint_as_float(q.w);
    return 4;
  }
}

__device__ __forceinline__ Lse2 lse2_add8(Lse2 st, const float* x, int n) {
  float cmax = -INFINITY;
  for (int e = 0; e < n; ++e) cmax = fmaxf(cmax, x[e] * kLog2e);
  const float M = fmaxf(st.m, cmax);
  float s = (st.m == -INFINITY) ? 0.f : st.s * exp2f(st.m - M);
  for (int e = 0; e < n; ++e) s += exp2f(fmaf(x[e], kLog2e, -M));
  return Lse2{M, s};
}

template <typename T>
__global__ void __launch_bounds__(kOvThreads) overlap_rows(const T* __restrict__ P,
                                                          const T* __restrict__ Q,
                                                          const int32_t* valid_len, int V,
                                                          int gamma, float* a_out, float* l1_out,
                                                          int* status) {
  constexpr int epc = 16 / (int)sizeof(T);
  __shared__ Lse2 red_p[kOvThreads / 32], red_q[kOvThreads / 32];
  __shared__ float red_a[kOvThreads / 32], red_l[kOvThreads / 32];
  __shared__ float s_lp, s_lq;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = blockIdx.x / gamma, i = blockIdx.x - n * gamma;
  int vl = valid_len[n];
  if (vl < 0 || vl > gamma) {
    if (tid == 0) set_status(status, kErrArg);
    vl = vl < 0 ? 0 : gamma;
  }
  if (i >= vl) {
    if (tid == 0) {
      a_out[blockIdx.x] = 0.f;
      l1_out[blockIdx.x] = 0.f;
    }
    return;
  }
  const T* prow = P + (size_t)blockIdx.x * V;
  const T* qrow = Q + (size_t)blockIdx.x * V;
  Lse2 sp = lse2_empty(), sq = lse2_empty();
  float x[8];
  for (int v0 = tid * epc; v0 < V; v0 += kOvThreads * epc) {
    const int ne = load_chunk(prow, v0, x);
    sp = lse2_add8(sp, x, ne);
    load_chunk(qrow, v0, x);
    sq = lse2_add8(sq, x, ne);
  }
  sp = warp_lse2(sp);
  sq = warp_lse2(sq);
  if (lane == 0) {
    red_p[warp] = sp;
    red_q[warp] = sq;
  }
  __syncthreads();
  if (tid == 0) {
    Lse2 lp = lse2_empty(), lq = lse2_empty();
    for (int w = 0; w < kOvThreads / 32; ++w) {
      lp = lse2_merge(lp, red_p[w]);
      lq = lse2_merge(lq, red_q[w]);
    }
    s_lp = lp.m + log2f(lp.s);   // base-2 log-normalisers of the scaled logits
    s_lq = lq.m + log2f(lq.s);
    if (!isfinite(s_lp) || !isfinite(s_lq)) set_status(status, kErrNonfinite);
  }
  __syncthreads();
  const float LP = s_lp, LQ = s_lq;
  float amin = 0.f, al1 = 0.f;
  float y[8];
  for (int v0 = tid * epc; v0 < V; v0 += kOvThreads * epc) {
    const int ne = load_chunk(prow, v0, x);
    load_chunk(qrow, v0, y);
    for (int e = 0; e < ne; ++e) {
      const float pv = exp2f(fmaf(x[e], kLog2e, -LP));
      const float qv = exp2f(fmaf(y[e], kLog2e, -LQ));
      amin += fminf(pv, qv);
      al1 += fabsf(pv - qv);
    }
  }
  amin = warp_sum(amin);
  al1 = warp_sum(al1);
  if (lane == 0) {
    red_a[warp] = amin;
    red_l[warp] = al1;
  }
  __syncthreads();
  if (tid == 0) {
    float sa = 0.f, sl = 0.f;
    for (int w = 0; w < kOvThreads / 32; ++w) {
      sa += red_a[w];
      sl += red_l[w];
    }
    a_out[blockIdx.x] = sa;
    l1_out[blockIdx.x] = sl;
  }
}

__global__ void __launch_bounds__(1024) overlap_finalize(const float* a, const int32_t* valid_len,
                                                         int N, int gamma, float* tau,
                                                         float* accept_rate, float* mean_tau) {
  __shared__ double red[32][2 * kMaxGamma + 2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  double sums[kMaxGamma], cnts[kMaxGamma];
  double tsum = 0.0, tcnt = 0.0;
  for (int i = 0; i < kMaxGamma; ++i) sums[i] = cnts[i] = 0.0;
  for (int n = tid; n < N; n += blockDim.x) {
    int vl = valid_len[n];
    vl = vl < 0 ? 0 : (vl > gamma ? gamma : vl);
    double acc = 1.0, t = 1.0;
    for (int i = 0; i < gamma; ++i) {
      const double ai = (double)a[(size_t)n * gamma + i];
      acc *= ai;
      t += acc;
      if (i < vl) {
        sums[i] += ai;
        cnts[i] += 1.0;
      }
    }
    tau[n] = (float)t;
    if (vl >= 1) {
      tsum += t;
      tcnt += 1.0;
    }
  }
  for (int i = 0; i < gamma; ++i) {
    sums[i] = warp_sum_f64(sums[i]);
    cnts[i] = warp_sum_f64(cnts[i]);
  }
  tsum = warp_sum_f64(tsum);
  tcnt = warp_sum_f64(tcnt);
  if (lane == 0) {
    for (int i = 0; i < gamma; ++i) {
      red[warp][i] = sums[i];
      red[warp][kMaxGamma + i] = cnts[i];
    }
    red[warp][2 * kMaxGamma] = tsum;
    red[warp][2 * kMaxGamma + 1] = tcnt;
  }
  __syncthreads();
  if (tid == 0) {
    const int nw = blockDim.x / 32;
    for (int i = 0; i < gamma; ++i) {
      double s = 0.0, c = 0.0;
      for (int w = 0; w < nw; ++w) {
        s += red[w][i];
        c += red[w][kMaxGamma + i];
      }
      accept_rate[i] = c > 0.0 ? (float)(s / c) : 0.f;
    }
    double s = 0.0, c = 0.0;
    for (int w = 0; w < nw; ++w) {
      s += red[w][2 * kMaxGamma];
      c += red[w][2 * kMaxGamma + 1];
    }
    *mean_tau = c > 0.0 ? (float)(s / c) : 0.f;
  }
}

cudaError_t launch_overlap(const Ctx& ctx, const OverlapArgs& a, cudaStream_t s) {
  if (a.N > 0) {
    const int grid = a.N * a.gamma;
    if (a.dtype == 1)
      overlap_rows<__nv_bfloat16><<<grid, kOvThreads, 0, s>>>(
          static_cast<const __nv_bfloat16*>(a.P), static_cast<const __nv_bfloat16*>(a.Q),
          a.valid_len, a.V, a.gamma, a.a, a.l1, ctx.ws.status);
    else
      overlap_rows<float><<<grid, kOvThreads, 0, s>>>(static_cast<const float*>(a.P),
                                                      static_cast<const float*>(a.Q), a.valid_len,
                                                      a.V, a.gamma, a.a, a.l1, ctx.ws.status);
    count_launch(ctx);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  overlap_finalize<<<1, 1024, 0, s>>>(a.a, a.valid_len, a.N, a.gamma, a.tau, a.accept_rate,
                                      a.mean_tau);
  count_launch(ctx);
  return cudaGetLastError();
}

}  // namespace dsd
