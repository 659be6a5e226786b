// Target-side rejection verification of the kept draft prefixes
// ("DeepSpec 训练全流程详解（以 Qwen3 + DSpark 为例）" 4.4 Verify;
// "DSpark 论文精读" 2.1 and 3.1).
//
// Kernels, in stream order:
//   verify_rows_build  one CTA: row list (r, t) for t = 0..keep_len[r] and the
//                      per-request row offsets (exclusive scan of keep_len+1).
//   verify_rows        persistent grid over (row, vocabulary split) items:
//                      streams only the B kept rows of P once (16-byte loads,
//                      evict-first), producing per split the base-2 lse of
//                      P/T and an argmax key (greedy: argmax P; sampled: the
//                      stream-3 Gumbel-max of the bonus row).
//   verify_decide      one warp per request: merges the splits, runs the
//                      accept tests in order and stops at the first
//                      rejection; writes accept_len and (unless a residual
//                      draw is needed) next_token.
//   residual pass      sampled only, requests with a rejection: recompute
//                      q_k from U, E, W (the CUDA-core bias path) and draw
//                      from norm(max(0, p_k - q_k)) by Gumbel-max (stream 2).
//   verify_finish      next_token of the rejected requests.
#include "dsd_common.cuh"

namespace dsd {

cudaError_t launch_residual_simt(const Ctx& ctx, const VerifyArgs& a, cudaStream_t s);

constexpr int kRowThreads = 256;

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__global__ void __launch_bounds__(1024) verify_rows_build(const int32_t* keep_len, int R, int gamma,
                                                          int2* rows, int* row_off, int* B_out,
                                                          int* status) {
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int IPT = (R + 1023) / 1024;
  const int r0 = tid * IPT;
  int local = 0;
  for (int t = 0; t < IPT; ++t) {
    const int r = r0 + t;
    if (r < R) {
      int L = keep_len[r];
      if (L < 0 || L > gamma) {
        set_status(status, kErrArg);
        L = L < 0 ? 0 : gamma;
      }
      local += L + 1;
    }
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = warp_tot[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_tot[lane] = wi - w;
    if (lane == 31) *B_out = wi;
  }
  __syncthreads();
  int off = warp_tot[warp] + incl - local;
  for (int t = 0; t < IPT; ++t) {
    const int r = r0 + t;
    if (r >= R) break;
    int L = keep_len[r];
    L = L < 0 ? 0 : (L > gamma ? gamma : L);
    row_off[r] = off;
    for (int q = 0; q <= L; ++q) rows[off + q] = make_int2(r, q);
    off += L + 1;
  }
}

struct RowsParams {
  int* status;
  const void* P;
  const int32_t* keep_len;
  const uint32_t* req_id;
  const int2* rows;
  const int* B;
  RowPart* parts;
  int V, gamma, chunk, sampled;
  float inv_T;
  uint32_t k0, k1;
};

// SAMPLED is p.sampled as a template argument, so the greedy rows (a
// running maximum only) get their own lean instantiation with more loads in
// flight.
template <typename T, bool SAMPLED>
__global__ void __launch_bounds__(kRowThreads) verify_rows(RowsParams p) {
  constexpr int epc = 16 / (int)sizeof(T);
  __shared__ Lse2 red_l[kRowThreads / 32];
  __shared__ unsigned long long red_k[kRowThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_items = (*p.B) * kVerifySplits;
  const T* P = static_cast<const T*>(p.P);
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int b = item / kVerifySplits, sp = item - b * kVerifySplits;
    const int2 rt = p.rows[b];
    const int r = rt.x, t = rt.y;
    int L = p.keep_len[r];
    L = L < 0 ? 0 : (L > p.gamma ? p.gamma : L);
    const bool bonus = (t == L);
    const uint32_t rid = p.req_id ? p.req_id[r] : (uint32_t)r;
    const T* row = P + ((size_t)r * (p.gamma + 1) + t) * p.V;
    const int v_begin = sp * p.chunk;
    const int v_end = min(p.V, v_begin + p.chunk);
    Lse2 st = lse2_empty();
    unsigned long long best = 0ull;
    // Greedy: running maximum value and its lowest index; a chunk's index is
    // looked up only when its maximum beats the running one.  NaN propagates
    // through max.NaN and is reported.
    float bz = -INFINITY;
    uint32_t bv = 0xFFFFFFFFu;
    bool nan_seen = false;
    const int v_first = v_begin + tid * epc;
    // Several 16-byte loads in flight per thread (eight for greedy rows,
    // four with the sampled path's larger register set): with one, the grid
    // keeps too few bytes in flight to cover the HBM latency.
    constexpr int kUnroll = SAMPLED ? 4 : 8;
    for (int vb = v_first; vb < v_end; vb += kUnroll * kRowThreads * epc) {
      uint4 q[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v0 = vb + u * kRowThreads * epc;
        q[u] = v0 < v_end ? ld_stream16(row + v0) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v0 = vb + u * kRowThreads * epc;
        if (v0 >= v_end) break;
        float x[8];
        if constexpr (sizeof(T) == 2) {
          x[0] = bf16lo(q[u].x); x[1] = bf16hi(q[u].x); x[2] = bf16lo(q[u].y); x[3] = bf16hi(q[u].y);
          x[4] = bf16lo(q[u].z); x[5] = bf16hi(q[u].z); x[6] = bf16lo(q[u].w); x[7] = bf16hi(q[u].w);
        } else {
          x[0] = __uint_as_float(q[u].x); x[1] = __uint_as_float(q[u].y);
          x[2] = __uint_as_float(q[u].z); x[3] = __uint_as_float(q[u].w);
        }
        if constexpr (!SAMPLED) {
          float m = max3_nan(x[0], x[1], x[2]);
#pragma unroll
          for (int e = 3; e < epc; e += 2)
            m = e + 1 < epc ? max3_nan(m, x[e], x[e + 1]) : max_nan(m, x[e]);
          if (!(m <= bz)) {          // a larger maximum, or NaN
            if (m != m) {
              nan_seen = true;
            } else {
              int idx = epc - 1;
#pragma unroll
              for (int e = epc - 2; e >= 0; --e)
                if (x[e] == m) idx = e;
              bz = m;
              bv = (uint32_t)(v0 + idx);
            }
          }
        } else {
          float cmax = -INFINITY;
#pragma unroll
          for (int e = 0; e < epc; ++e) {
            x[e] *= p.inv_T;
            cmax = fmaxf(cmax, x[e] * kLog2e);
          }
          const float M = fmaxf(st.m, cmax);
          float s = st.s * exp2f(st.m - M);
#pragma unroll
          for (int e = 0; e < epc; ++e) s += exp2f(fmaf(x[e], kLog2e, -M));
          st.m = M;
          st.s = s;
          if (bonus) {
#pragma unroll
            for (int e = 0; e < epc; e += 4) {
              const uint32_t v = (uint32_t)(v0 + e);
              const Philox4 ph = philox4x32_10(v >> 2, (uint32_t)t, rid, 3u, p.k0, p.k1);
              // v0 is a multiple of 4 (epc-aligned), so words map to v .. v+3
              const float z0 = x[e + 0] + gumbel_from_word(ph.x);
              const float z1 = x[e + 1] + gumbel_from_word(ph.y);
              const float z2 = x[e + 2] + gumbel_from_word(ph.z);
              const float z3 = x[e + 3] + gumbel_from_word(ph.w);
              unsigned long long k;
              k = make_key(z0, v + 0); best = k > best ? k : best;
              k = make_key(z1, v + 1); best = k > best ? k : best;
              k = make_key(z2, v + 2); best = k > best ? k : best;
              k = make_key(z3, v + 3); best = k > best ? k : best;
            }
          }
        }
      }
    }
    if (!SAMPLED && v_first < v_end) {
      if (nan_seen) set_status(p.status, kErrNonfinite);
      // every element was -inf: the first one holds the maximum
      best = make_key(bz, bv == 0xFFFFFFFFu ? (uint32_t)v_first : bv);
    }
    if constexpr (SAMPLED) st = warp_lse2(st);   // greedy rows have no normaliser
    best = warp_max_u64(best);
    if (lane == 0) {
      red_l[warp] = st;
      red_k[warp] = best;
    }
    __syncthreads();
    if (tid == 0) {
      Lse2 l = lse2_empty();
      unsigned long long k = 0ull;
      for (int w = 0; w < kRowThreads / 32; ++w) {
        if constexpr (SAMPLED) l = lse2_merge(l, red_l[w]);
        k = red_k[w] > k ? red_k[w] : k;
      }
      p.parts[item] = RowPart{l.m, l.s, k};
    }
    __syncthreads();
  }
}

struct DecideParams {
  const void* P;
  const int32_t* tokens;
  const float* lse_q;
  const float* logit_at_tok;
  const int32_t* keep_len;
  const uint32_t* req_id;
  const int* row_off;
  const RowPart* parts;
  int32_t* accept_len;
  int32_t* next_token;
  int* rej_list;
  int* rej_k;
  float* rej_lseP;
  unsigned int* n_rej;
  int* status;
  int R, V, gamma, sampled;
  float inv_T;
  uint32_t k0, k1;
};

template <typename T>
__global__ void __launch_bounds__(256) verify_decide(DecideParams p) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= p.R) return;
  const T* P = static_cast<const T*>(p.P);
  int L = p.keep_len[r];
  L = L < 0 ? 0 : (L > p.gamma ? p.gamma : L);
  const int off = p.row_off[r];
  const uint32_t rid = p.req_id ? p.req_id[r] : (uint32_t)r;
  int k = L;
  float lseP_k = 0.f;
  for (int t = 0; t < L; ++t) {
    // merge the splits of row t (lanes 0..kVerifySplits-1)
    Lse2 l = lse2_empty();
    unsigned long long key = 0ull;
    if (lane < kVerifySplits) {
      const RowPart rp = p.parts[(size_t)(off + t) * kVerifySplits + lane];
      l = Lse2{rp.m, rp.s};
      key = rp.key;
    }
    l = warp_lse2(l);
    key = warp_max_u64(key);
    int x = p.tokens[(size_t)r * p.gamma + t];
    bool ok;
    if (!p.sampled) {
      ok = (int)key_index(key) == x;
    } else {
      if (x < 0 || x >= p.V) {
        set_status(p.status, kErrArg);
        x = 0;
      }
      const float lseP = lse2_value(l);
      const float pl = ld_elem(P, ((size_t)r * (p.gamma + 1) + t) * p.V + x) * p.inv_T - lseP;
      const float ql = p.logit_at_tok[(size_t)r * p.gamma + t] - p.lse_q[(size_t)r * p.gamma + t];
      const float lr = pl - ql;
      const float accept_prob = lr >= 0.f ? 1.f : __expf(lr);
      const Philox4 ph = philox4x32_10(0u, (uint32_t)t, rid, 1u, p.k0, p.k1);
      const float u = uniform_from_word(ph.x);
      ok = u < accept_prob;
      if (!isfinite(lseP) || !isfinite(ql)) set_status(p.status, kErrNonfinite);
      lseP_k = lseP;
    }
    if (!ok) {
      k = t;
      break;
    }
  }
  int next = -1;
  if (!p.sampled || k == L) {
    unsigned long long key = 0ull;
    if (lane < kVerifySplits) key = p.parts[(size_t)(off + k) * kVerifySplits + lane].key;
    key = warp_max_u64(key);
    next = (int)key_index(key);
    if (key == 0ull) set_status(p.status, kErrNonfinite);
  } else if (lane == 0) {
    const unsigned int slot = atomicAdd(p.n_rej, 1u);
    p.rej_list[slot] = r;
    p.rej_k[r] = k;
    p.rej_lseP[r] = lseP_k;
  }
  if (lane == 0) {
    p.accept_len[r] = k;
    p.next_token[r] = next;
  }
}

__global__ void verify_finish(const int* rej_list, const unsigned int* n_rej,
                              const unsigned long long* res_keys, const float* res_sums, int R_max,
                              int32_t* next_token, int* status) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int)*n_rej) return;
  const int r = rej_list[i];
  const float res = res_sums[r], psum = res_sums[R_max + r];
  // An empty residual (p ~ q everywhere) falls back to sampling p itself.
  const unsigned long long key = (res > 1e-12f * psum && res_keys[r]) ? res_keys[r] : res_keys[R_max + r];
  if (key == 0ull) set_status(status, kErrNonfinite);
  next_token[r] = (int32_t)key_index(key);
}

cudaError_t launch_verify(const Ctx& ctx, const VerifyArgs& a, cudaStream_t s) {
  const Workspace& ws = ctx.ws;
  const int sampled = a.temperature > 0.f ? 1 : 0;
  const float inv_T = sampled ? 1.f / a.temperature : 1.f;
  const uint32_t k0 = (uint32_t)(a.seed & 0xFFFFFFFFull), k1 = (uint32_t)(a.seed >> 32);
  int* row_off = ws.rej_k + ctx.cfg.R_max;  // carved next to rej_k
  cudaError_t e = cudaMemsetAsync(ws.counters, 0, 16 * sizeof(unsigned int), s);
  if (e != cudaSuccess) return e;
  if (sampled) {
    e = cudaMemsetAsync(ws.res_keys, 0, 2 * sizeof(unsigned long long) * ctx.cfg.R_max, s);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(ws.res_sums, 0, 2 * sizeof(float) * ctx.cfg.R_max, s);
    if (e != cudaSuccess) return e;
  }
  verify_rows_build<<<1, 1024, 0, s>>>(a.keep_len, a.R, a.gamma, ws.rows, row_off, ws.sched_B,
                                       ws.status);
  count_launch(ctx);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  RowsParams rp{};
  rp.status = ws.status;
  rp.P = a.P;
  rp.keep_len = a.keep_len;
  rp.req_id = a.req_id;
  rp.rows = ws.rows;
  rp.B = ws.sched_B;
  rp.parts = ws.vparts;
  rp.V = a.V;
  rp.gamma = a.gamma;
  const int epc = ctx.cfg.dtype == 1 ? 8 : 4;
  int chunk = (a.V + kVerifySplits - 1) / kVerifySplits;
  chunk = (chunk + epc - 1) / epc * epc;
  rp.chunk = chunk;
  rp.sampled = sampled;
  rp.inv_T = inv_T;
  rp.k0 = k0;
  rp.k1 = k1;
  const int grid_rows = ctx.num_sms * 4;
  if (ctx.cfg.dtype == 1) {
    if (sampled)
      verify_rows<__nv_bfloat16, true><<<grid_rows, kRowThreads, 0, s>>>(rp);
    else
      verify_rows<__nv_bfloat16, false><<<grid_rows, kRowThreads, 0, s>>>(rp);
  } else {
    if (sampled)
      verify_rows<float, true><<<grid_rows, kRowThreads, 0, s>>>(rp);
    else
      verify_rows<float, false><<<grid_rows, kRowThreads, 0, s>>>(rp);
  }
  count_launch(ctx);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  DecideParams dp{};
  dp.P = a.P;
  dp.tokens = a.tokens;
  dp.lse_q = a.lse_q;
  dp.logit_at_tok = a.logit_at_tok;
  dp.keep_len = a.keep_len;
  dp.req_id = a.req_id;
  dp.row_off = row_off;
  dp.parts = ws.vparts;
  dp.accept_len = a.accept_len;
  dp.next_token = a.next_token;
  dp.rej_list = ws.rej_list;
  dp.rej_k = ws.rej_k;
  dp.rej_lseP = ws.rej_lseP;
  dp.n_rej = ws.counters + 1;
  dp.status = ws.status;
  dp.R = a.R;
  dp.V = a.V;
  dp.gamma = a.gamma;
  dp.sampled = sampled;
  dp.inv_T = inv_T;
  dp.k0 = k0;
  dp.k1 = k1;
  const int grid_dec = (a.R + 7) / 8;
  if (ctx.cfg.dtype == 1)
    verify_decide<__nv_bfloat16><<<grid_dec, 256, 0, s>>>(dp);
  else
    verify_decide<float><<<grid_dec, 256, 0, s>>>(dp);
  count_launch(ctx);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  if (sampled) {
    e = launch_residual_simt(ctx, a, s);
    if (e != cudaSuccess) return e;
    verify_finish<<<(a.R + 255) / 256, 256, 0, s>>>(ws.rej_list, ws.counters + 1, ws.res_keys,
                                                    ws.res_sums, ctx.cfg.R_max, a.next_token,
                                                    ws.status);
    count_launch(ctx);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dsd
