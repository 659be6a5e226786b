// CUDA-core path of the Markov-head bias projection (the GEMV path for small
// batches and fp32 tables), used by dsd_propose (one launch per draft
// position) and by dsd_verify's residual pass.
//
// Pages: "Qwen3.8-Flash-Next DSpark 训练实验", Baseline 架构 / Markov 顺序修正
// (m_i = W_1[t_{i-1}], b_i = W_2 m_i, l_i = l_i^0 + b_i, argmax over the full
// vocabulary); "DSpark 论文精读" 2.2 (x_j ~ Softmax(U_j + b)); "DeepSpec 训练全
// 流程详解" 4.4 (residual resampling).
//
// Work split: the vocabulary is cut into 128-row tiles of W ([V, r] layout,
// so a tile is one contiguous block of memory); CTAs stride over tiles.  A CTA
// stages the W tile in shared memory (16-byte chunks XOR-swizzled by row so
// that eight consecutive rows read by a quarter-warp hit distinct banks) and
// the gathered rows m = act(E[prev]) of up to 16 requests in fp32.  Thread
// (vp, qq) owns vocabulary entries v0 + vp and v0 + vp + 64 and requests
// 4 qq .. 4 qq + 3, so each 16-byte chunk of W read from shared memory feeds
// four requests and each chunk of a Markov row two vocabulary entries; it
// computes the 8 bias values, adds U and folds each biased logit into a
// running base-2 log-sum-exp and a packed argmax key per request.  The
// biased logits never leave registers.  At the end the CTA reduces per
// request and publishes one atomicMax key and one (m, s) partial per
// request.
#include "dsd_common.cuh"
#include "schedule.cuh"
#include "tc_ptx.cuh"

namespace dsd {

constexpr int kSimtThreads = 256;
constexpr int kSimtTileV = 128;
constexpr int kSimtRC = 16;   // requests per pass
constexpr int kSimtRPT = 4;   // requests per thread
constexpr int kSimtRows = 2;  // vocabulary rows per thread (vp and vp + kSimtTileV / 2)
constexpr int kSimtHalfV = kSimtTileV / kSimtRows;
static_assert(kSimtThreads == kSimtHalfV * (kSimtRC / kSimtRPT), "thread = (row pair, request group)");
static_assert(kSimtRPT == 4 && kSimtHalfV % 4 == 0, "a quad of lanes shares one Philox block per request");

enum SimtMode { kModeStep = 0, kModeResidual = 1 };

struct SimtParams {
  const void* U;
  const void* E;
  const void* W;
  const void* P;                 // residual mode: target logits [R, gamma+1, V]
  const int32_t* prev_tok;
  const int32_t* tokens;         // residual mode: draft tokens [R, gamma]
  const uint32_t* req_id;
  const float* lse_q;            // residual mode
  const float* A;                // gated head: [R, gamma, rank] representations (else nullptr)
  unsigned long long* cand_parts;  // candidate lists: [gamma][n_part][cand_R][kCandK] keys
  int cand, cand_R;              // step mode: also keep the CTA's top-kCandK per request
  unsigned long long* keys;      // step: [gamma][R_max]; residual: [2][R_max]
  float2* parts;                 // step: [gamma][n_part][R_max]
  float* res_sums;               // residual: [2][R_max]
  const int* rej_list;           // residual: request list
  const int* rej_k;              // residual: rejection position per request
  const float* rej_lseP;         // residual: target lse (natural) per request
  const unsigned int* n_rej;     // residual: number of listed requests
  int* status;
  int R, R_max, V, rank, gamma, j, act, bias_at_first, swz_mask, n_part;
  float inv_T;
  int sampled;
  uint32_t k0, k1;
};

// 16-byte asynchronous copy global -> shared with an L2 cache policy, and
// the wait for all of this thread's copies.
__device__ __forceinline__ void cp_async_keep16(void* dst, const void* src, uint64_t pol) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(d), "l"(src),
               "l"(pol)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

template <typename T>
__device__ __forceinline__ int unpack16(const uint4& q, float* w) {
  if constexpr (sizeof(T) == 2) {
    w[0] = bf16lo(q.x); w[1] = bf16hi(q.x); w[2] = bf16lo(q.y); w[3] = bf16hi(q.y);
    w[4] = bf16lo(q.z); w[5] = bf16hi(q.z); w[6] = bf16lo(q.w); w[7] = bf16hi(q.w);
    return 8;
  } else {
    w[0] = __uint_as_float(q.x); w[1] = __uint_as_float(q.y);
    w[2] = __uint_as_float(q.z); w[3] = __uint_as_float(q.w);
    return 4;
  }
}

// Candidate lists of one CTA: per request a sorted top-kCandK of packed
// (biased logit, token) keys, a threshold (its kCandK-th key, or 0 while it
// is not full) and an append buffer for one tile (at most kSimtTileV keys).
// One warp merges a request's buffer into its list: kCandK rounds of a
// warp-wide maximum over the list and the buffer (keys are unique: the token
// index is part of the key).
__device__ __forceinline__ void cand_merge(unsigned long long* list, unsigned long long* buf,
                                           unsigned long long* thr, int* cnt, int nr, int warp,
                                           int lane) {
  for (int rr = warp; rr < nr; rr += kSimtThreads / 32) {
    const int n = cnt[rr];
    if (n == 0) continue;
    unsigned long long k[1 + kSimtTileV / 32];
    k[0] = lane < kCandK ? list[rr * kCandK + lane] : 0ull;
#pragma unroll
    for (int q = 0; q < kSimtTileV / 32; ++q) {
      const int i = lane + 32 * q;
      k[q + 1] = i < n ? buf[rr * kSimtTileV + i] : 0ull;
    }
    __syncwarp();
    for (int t = 0; t < kCandK; ++t) {
      unsigned long long m = 0ull;
#pragma unroll
      for (int q = 0; q < 1 + kSimtTileV / 32; ++q) m = k[q] > m ? k[q] : m;
      const unsigned long long wm = warp_max_u64(m);
      if (wm != 0ull && m == wm) {
#pragma unroll
        for (int q = 0; q < 1 + kSimtTileV / 32; ++q)
          if (k[q] == wm) k[q] = 0ull;
      }
      if (lane == 0) list[rr * kCandK + t] = wm;
    }
    __syncwarp();
    if (lane == 0) {
      thr[rr] = list[rr * kCandK + kCandK - 1];
      cnt[rr] = 0;
    }
  }
}

template <typename T, int MODE>
__global__ void __launch_bounds__(kSimtThreads) simt_bias_kernel(SimtParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int epc = 16 / (int)sizeof(T);
  const int rank = p.rank;
  const int nch = rank / epc;
  // Markov rows of request pairs interleaved: pair pp holds element k of
  // requests 2 pp and 2 pp + 1 side by side, so one 8-byte word feeds both
  // halves of a packed fp32x2 FMA
  const int mstride2 = 2 * rank + 8;
  unsigned char* Ws = smem;
  float* ms = reinterpret_cast<float*>(smem + (size_t)kSimtTileV * nch * 16);
  // candidate lists (step mode with p.cand), after ms
  unsigned long long* c_list = reinterpret_cast<unsigned long long*>(ms + (size_t)(kSimtRC / 2) * mstride2);
  unsigned long long* c_buf = c_list + kSimtRC * kCandK;
  unsigned long long* c_thr = c_buf + kSimtRC * kSimtTileV;
  int* c_cnt = reinterpret_cast<int*>(c_thr + kSimtRC);
  const bool cand = (MODE == kModeStep) && p.cand;

  __shared__ int s_prev[kSimtRC];
  __shared__ int s_req[kSimtRC];
  __shared__ int s_row[kSimtRC];       // row of U (r*gamma + position)
  __shared__ int s_bias[kSimtRC];
  __shared__ float s_lseq[kSimtRC];
  __shared__ float s_lsep[kSimtRC];
  __shared__ uint32_t s_rid[kSimtRC];
  __shared__ int s_pos[kSimtRC];
  __shared__ Lse2 red_l[8][kSimtRPT];
  __shared__ unsigned long long red_k[8][kSimtRPT];
  __shared__ unsigned long long red_k2[8][kSimtRPT];
  __shared__ float red_f[8][kSimtRPT];
  __shared__ float red_f2[8][kSimtRPT];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // thread = vocabulary rows vp and vp + 64 of the tile x requests
  // 4 qq .. 4 qq + 3: each 16-byte chunk of a W row read from shared memory
  // feeds four requests, each chunk of a Markov row two vocabulary rows
  const int vp = tid & (kSimtHalfV - 1), qq = tid / kSimtHalfV;
  const int ntiles = (p.V + kSimtTileV - 1) / kSimtTileV;
  const T* U = static_cast<const T*>(p.U);
  const T* E = static_cast<const T*>(p.E);
  const T* W = static_cast<const T*>(p.W);
  const T* P = static_cast<const T*>(p.P);

  const int nreq = (MODE == kModeStep) ? p.R : (int)min(*p.n_rej, (unsigned)p.R);

  for (int r0 = 0; r0 < nreq; r0 += kSimtRC) {
    const int nr = min(kSimtRC, nreq - r0);
    __syncthreads();
    if (tid < kSimtRC) {
      int prev = 0, req = 0, row = 0, bias = 0, pos = 0;
      float lq = 0.f, lp = 0.f;
      if (tid < nr) {
        if constexpr (MODE == kModeStep) {
          req = r0 + tid;
          pos = p.j;
          prev = (p.j == 0) ? p.prev_tok[req]
                            : (int)key_index(p.keys[(size_t)(p.j - 1) * p.R_max + req]);
        } else {
          req = p.rej_list[r0 + tid];
          pos = p.rej_k[req];
          prev = (pos == 0) ? p.prev_tok[req] : p.tokens[(size_t)req * p.gamma + pos - 1];
          lq = p.lse_q[(size_t)req * p.gamma + pos];
          lp = p.rej_lseP[req];
        }
        if (prev < 0 || prev >= p.V) {
          set_status(p.status, kErrArg);
          prev = 0;
        }
        bias = (pos > 0 || p.bias_at_first) ? 1 : 0;
        row = req * p.gamma + pos;
      }
      s_prev[tid] = prev;
      s_req[tid] = req;
      s_row[tid] = row;
      s_bias[tid] = bias;
      s_lseq[tid] = lq;
      s_lsep[tid] = lp;
      s_pos[tid] = pos;
      s_rid[tid] = p.req_id ? p.req_id[req] : (uint32_t)req;
    }
    __syncthreads();
    // the Markov rows (or the head's representations), 16 bytes per load
    if (p.A) {
      for (int idx = tid; idx < (kSimtRC / 2) * (rank / 4); idx += kSimtThreads) {
        const int pp = idx / (rank / 4), k = (idx - pp * (rank / 4)) * 4;
        float4 m[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int rr = 2 * pp + h;
          m[h] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (rr < nr && s_bias[rr])
            m[h] = __ldg(reinterpret_cast<const float4*>(
                p.A + ((size_t)s_req[rr] * p.gamma + s_pos[rr]) * rank + k));
        }
        float4* dst = reinterpret_cast<float4*>(ms + pp * mstride2 + 2 * k);
        dst[0] = make_float4(m[0].x, m[1].x, m[0].y, m[1].y);
        dst[1] = make_float4(m[0].z, m[1].z, m[0].w, m[1].w);
      }
    } else {
      for (int idx = tid; idx < (kSimtRC / 2) * nch; idx += kSimtThreads) {
        const int pp = idx / nch, k = (idx - pp * nch) * epc;
        float m[2][8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int rr = 2 * pp + h;
#pragma unroll
          for (int e = 0; e < 8; ++e) m[h][e] = 0.f;
          if (rr < nr && s_bias[rr]) {
            unpack16<T>(ld_keep16(E + (size_t)s_prev[rr] * rank + k), m[h]);
#pragma unroll
            for (int e = 0; e < epc; ++e) m[h][e] = act_apply(m[h][e], p.act);
          }
        }
        float4* dst = reinterpret_cast<float4*>(ms + pp * mstride2 + 2 * k);
#pragma unroll
        for (int e = 0; e < epc; e += 2) dst[e / 2] = make_float4(m[0][e], m[1][e], m[0][e + 1], m[1][e + 1]);
      }
    }
    if (cand) {
      for (int i = tid; i < kSimtRC * kCandK; i += kSimtThreads) c_list[i] = 0ull;
      if (tid < kSimtRC) {
        c_thr[tid] = 0ull;
        c_cnt[tid] = 0;
      }
    }

    Lse2 st[kSimtRPT];
    unsigned long long best[kSimtRPT], best2[kSimtRPT];
    float fsum[kSimtRPT], fsum2[kSimtRPT];
#pragma unroll
    for (int i = 0; i < kSimtRPT; ++i) {
      st[i] = lse2_empty();
      best[i] = 0ull;
      best2[i] = 0ull;
      fsum[i] = 0.f;
      fsum2[i] = 0.f;
    }

    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const int v0 = tile * kSimtTileV;
      __syncthreads();
      if (cand) cand_merge(c_list, c_buf, c_thr, c_cnt, nr, warp, lane);   // the previous tile's
      // the W tile by asynchronous 16-byte copies: all of them in flight at
      // once, no registers held (rows past V are zero-filled)
      const int total = kSimtTileV * nch;
      const uint64_t pol = policy_evict_last();
      for (int c = tid; c < total; c += kSimtThreads) {
        const int row = c / nch, ch = c - row * nch;
        const int v = v0 + row;
        unsigned char* dst = Ws + ((size_t)row * nch + (ch ^ (row & p.swz_mask))) * 16;
        if (v < p.V)
          cp_async_keep16(dst, W + (size_t)v * rank + ch * epc, pol);
        else
          *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      }
      // this thread's U (and, residual, P) entries of the tile, loaded while
      // the W copies are in flight
      float uval[kSimtRows][kSimtRPT], pval[kSimtRows][kSimtRPT];
#pragma unroll
      for (int rho = 0; rho < kSimtRows; ++rho) {
        const int v = v0 + vp + rho * kSimtHalfV;
#pragma unroll
        for (int i = 0; i < kSimtRPT; ++i) {
          const int rr = qq * kSimtRPT + i;
          const bool ok = rr < nr && v < p.V;
          uval[rho][i] = ok ? ld_elem(U, (size_t)s_row[rr] * p.V + v) : 0.f;
          pval[rho][i] = 0.f;
          if constexpr (MODE == kModeResidual)
            if (ok)
              pval[rho][i] = ld_elem(P, ((size_t)s_req[rr] * (p.gamma + 1) + s_pos[rr]) * p.V + v);
        }
      }
      // the Philox words of this thread's Gumbel noise, also computed while
      // the W copies are in flight.  The four lanes of a quad hold four
      // consecutive vocabulary entries, which share one Philox block per
      // request: lane d of the quad computes the block of request 4 qq + d
      // and the quad hands the words round by shuffles (every lane takes
      // part, so this comes before any lane leaves the tile).
      uint32_t nword[kSimtRows][kSimtRPT];
      if (MODE == kModeResidual || p.sampled) {
        const int d = lane & 3, qbase = lane & ~3;
        const int rr_d = qq * kSimtRPT + d;
        const uint32_t c1 = (MODE == kModeResidual) ? (uint32_t)s_pos[rr_d] : (uint32_t)p.j;
        const uint32_t c3 = (MODE == kModeResidual) ? 2u : 0u;
#pragma unroll
        for (int rho = 0; rho < kSimtRows; ++rho) {
          const uint32_t v = (uint32_t)(v0 + vp + rho * kSimtHalfV);
          const Philox4 ph = philox4x32_10(v >> 2, c1, s_rid[rr_d], c3, p.k0, p.k1);
#pragma unroll
          for (int i = 0; i < kSimtRPT; ++i) {
            const uint32_t x = __shfl_sync(0xffffffffu, ph.x, qbase + i);
            const uint32_t y = __shfl_sync(0xffffffffu, ph.y, qbase + i);
            const uint32_t z = __shfl_sync(0xffffffffu, ph.z, qbase + i);
            const uint32_t w = __shfl_sync(0xffffffffu, ph.w, qbase + i);
            nword[rho][i] = d == 0 ? x : (d == 1 ? y : (d == 2 ? z : w));
          }
        }
      }
      cp_async_wait();
      __syncthreads();
      if (v0 + vp >= p.V) continue;   // both rows past the vocabulary
      // accumulators of request pairs: one packed fp32x2 FMA per W element
      // and pair (each half rounds as a scalar fmaf would)
      uint64_t acc2[kSimtRows][kSimtRPT / 2];
#pragma unroll
      for (int rho = 0; rho < kSimtRows; ++rho)
#pragma unroll
        for (int h = 0; h < kSimtRPT / 2; ++h) acc2[rho][h] = 0ull;
      const int r1 = vp + kSimtHalfV;
      const unsigned char* wrow0 = Ws + (size_t)vp * nch * 16;
      const unsigned char* wrow1 = Ws + (size_t)r1 * nch * 16;
      const float* mbase = ms + (qq * (kSimtRPT / 2)) * mstride2;
      for (int ch = 0; ch < nch; ++ch) {
        const uint4 q0 = *reinterpret_cast<const uint4*>(wrow0 + (ch ^ (vp & p.swz_mask)) * 16);
        const uint4 q1 = *reinterpret_cast<const uint4*>(wrow1 + (ch ^ (r1 & p.swz_mask)) * 16);
        float w0[8], w1[8];
        unpack16<T>(q0, w0);
        unpack16<T>(q1, w1);
#pragma unroll
        for (int h = 0; h < kSimtRPT / 2; ++h) {
          const ulonglong2* mrow =
              reinterpret_cast<const ulonglong2*>(mbase + h * mstride2 + ch * epc * 2);
#pragma unroll
          for (int e2 = 0; e2 < epc / 2; ++e2) {
            const ulonglong2 m2 = mrow[e2];
            acc2[0][h] = tc::fma2(tc::pack2(w0[2 * e2], w0[2 * e2]), m2.x, acc2[0][h]);
            acc2[1][h] = tc::fma2(tc::pack2(w1[2 * e2], w1[2 * e2]), m2.x, acc2[1][h]);
            acc2[0][h] = tc::fma2(tc::pack2(w0[2 * e2 + 1], w0[2 * e2 + 1]), m2.y, acc2[0][h]);
            acc2[1][h] = tc::fma2(tc::pack2(w1[2 * e2 + 1], w1[2 * e2 + 1]), m2.y, acc2[1][h]);
          }
        }
      }
      float acc[kSimtRows][kSimtRPT];
#pragma unroll
      for (int rho = 0; rho < kSimtRows; ++rho)
#pragma unroll
        for (int h = 0; h < kSimtRPT / 2; ++h) tc::unpack2(acc2[rho][h], acc[rho][2 * h], acc[rho][2 * h + 1]);
#pragma unroll
      for (int rho = 0; rho < kSimtRows; ++rho)
#pragma unroll
      for (int i = 0; i < kSimtRPT; ++i) {
        const int v = v0 + vp + rho * kSimtHalfV;
        const int rr = qq * kSimtRPT + i;
        if (rr >= nr || v >= p.V) continue;
        const float x = acc[rho][i] + uval[rho][i];
        if constexpr (MODE == kModeStep) {
          if (cand) {
            const unsigned long long ck = make_key(x, (uint32_t)v);
            if (ck > c_thr[rr]) c_buf[rr * kSimtTileV + atomicAdd(&c_cnt[rr], 1)] = ck;
          }
          const float xs = p.sampled ? x * p.inv_T : x;
          const float x2 = xs * kLog2e;
          const float M = fmaxf(st[i].m, x2);
          st[i].s = st[i].s * exp2f(st[i].m - M) + exp2f(x2 - M);
          st[i].m = M;
          float z = xs;
          if (p.sampled) z += gumbel_from_word(nword[rho][i]);
          const unsigned long long key = make_key(z, (uint32_t)v);
          best[i] = key > best[i] ? key : best[i];
        } else {
          // residual: res = max(0, p - q) with q = exp(l/T - lse_q), p = exp(P/T - lseP)
          const float pl = pval[rho][i] * p.inv_T - s_lsep[rr];
          const float ql = x * p.inv_T - s_lseq[rr];
          const float pv = __expf(pl);
          const float qv = __expf(ql);
          const float g = gumbel_from_word(nword[rho][i]);
          if (pl > ql) {
            // log(p - q) = pl + log(1 - exp(ql - pl)), kept accurate when p ~ q
            const float lr = pl + log2_one_minus_exp2((ql - pl) * kLog2e) * kLn2;
            const unsigned long long key = make_key(lr + g, (uint32_t)v);
            best[i] = key > best[i] ? key : best[i];
            fsum[i] += pv - qv;
          }
          const unsigned long long key2 = make_key(pl + g, (uint32_t)v);
          best2[i] = key2 > best2[i] ? key2 : best2[i];
          fsum2[i] += pv;
        }
      }
    }

    // CTA reduction per request: the two warps of its request group.
#pragma unroll
    for (int i = 0; i < kSimtRPT; ++i) {
      const Lse2 l = warp_lse2(st[i]);
      const unsigned long long k = warp_max_u64(best[i]);
      const unsigned long long k2 = warp_max_u64(best2[i]);
      const float f = warp_sum(fsum[i]);
      const float f2 = warp_sum(fsum2[i]);
      if (lane == 0) {
        red_l[warp][i] = l;
        red_k[warp][i] = k;
        red_k2[warp][i] = k2;
        red_f[warp][i] = f;
        red_f2[warp][i] = f2;
      }
    }
    __syncthreads();
    if (tid < kSimtRC && tid < nr) {
      const int g = tid / kSimtRPT, i = tid % kSimtRPT;
      constexpr int kWarpsPerGroup = kSimtHalfV / 32;
      Lse2 l = lse2_empty();
      unsigned long long k = 0ull, k2 = 0ull;
      float f = 0.f, f2 = 0.f;
      for (int w = g * kWarpsPerGroup; w < (g + 1) * kWarpsPerGroup; ++w) {
        l = lse2_merge(l, red_l[w][i]);
        k = red_k[w][i] > k ? red_k[w][i] : k;
        k2 = red_k2[w][i] > k2 ? red_k2[w][i] : k2;
        f += red_f[w][i];
        f2 += red_f2[w][i];
      }
      const int req = s_req[tid];
      if constexpr (MODE == kModeStep) {
        if (k) atomicMax(&p.keys[(size_t)p.j * p.R_max + req], k);
        p.parts[((size_t)p.j * p.n_part + blockIdx.x) * p.R_max + req] = make_float2(l.m, l.s);
      } else {
        if (k) atomicMax(&p.keys[req], k);
        if (k2) atomicMax(&p.keys[p.R_max + req], k2);
        atomicAdd(&p.res_sums[req], f);
        atomicAdd(&p.res_sums[p.R_max + req], f2);
      }
    }
    if (cand) {   // the last tile's candidates, then this CTA's lists
      __syncthreads();
      cand_merge(c_list, c_buf, c_thr, c_cnt, nr, warp, lane);
      __syncthreads();
      for (int i = tid; i < nr * kCandK; i += kSimtThreads) {
        const int rr = i / kCandK, q = i - rr * kCandK;
        p.cand_parts[(((size_t)p.j * p.n_part + blockIdx.x) * p.cand_R + s_req[rr]) * kCandK + q] =
            c_list[i];
      }
    }
  }
}

static size_t simt_smem_bytes(int rank, int elem_bytes, bool cand) {
  size_t b = (size_t)kSimtTileV * rank * elem_bytes + (size_t)kSimtRC * (rank + 4) * sizeof(float);
  if (cand)
    b += sizeof(unsigned long long) * ((size_t)kSimtRC * (kCandK + kSimtTileV + 1)) +
         sizeof(int) * kSimtRC;
  return b;
}

template <typename T, int MODE>
static cudaError_t launch_simt_typed(const SimtParams& sp, int grid, cudaStream_t s) {
  const size_t smem = simt_smem_bytes(sp.rank, (int)sizeof(T), MODE == kModeStep && sp.cand);
  cudaError_t e = cudaFuncSetAttribute(simt_bias_kernel<T, MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  simt_bias_kernel<T, MODE><<<grid, kSimtThreads, smem, s>>>(sp);
  return cudaGetLastError();
}

static cudaError_t launch_simt(const SimtParams& sp, int dtype, int grid, cudaStream_t s, int mode) {
  if (dtype == 1) {
    return mode == kModeStep ? launch_simt_typed<__nv_bfloat16, kModeStep>(sp, grid, s)
                             : launch_simt_typed<__nv_bfloat16, kModeResidual>(sp, grid, s);
  }
  return mode == kModeStep ? launch_simt_typed<float, kModeStep>(sp, grid, s)
                           : launch_simt_typed<float, kModeResidual>(sp, grid, s);
}

static SimtParams base_params(const Ctx& ctx, int R, int V, int rank, int gamma, int act,
                              int bias_at_first, float temperature, uint64_t seed) {
  SimtParams sp{};
  sp.status = ctx.ws.status;
  sp.R = R;
  sp.R_max = ctx.cfg.R_max;
  sp.V = V;
  sp.rank = rank;
  sp.gamma = gamma;
  sp.act = act;
  sp.bias_at_first = bias_at_first;
  sp.swz_mask = chunk_swizzle_mask(rank * (ctx.cfg.dtype == 1 ? 2 : 4) / 16);
  sp.n_part = ctx.n_part;
  sp.sampled = temperature > 0.f ? 1 : 0;
  sp.inv_T = temperature > 0.f ? 1.f / temperature : 1.f;
  sp.k0 = (uint32_t)(seed & 0xFFFFFFFFull);
  sp.k1 = (uint32_t)(seed >> 32);
  return sp;
}

int simt_grid(const Ctx& ctx, int V) {
  const int ntiles = (V + kSimtTileV - 1) / kSimtTileV;
  return ntiles < ctx.n_part ? ntiles : ctx.n_part;
}

cudaError_t launch_propose_simt(const Ctx& ctx, const ProposeArgs& a, cudaStream_t s) {
  SimtParams sp = base_params(ctx, a.R, a.V, a.rank, a.gamma, a.act, a.bias_at_first,
                              a.temperature, a.seed);
  sp.U = a.U;
  sp.E = a.E;
  sp.W = a.W;
  sp.prev_tok = a.prev_tok;
  sp.req_id = a.req_id;
  sp.keys = ctx.ws.keys;
  sp.parts = ctx.ws.lse_parts;
  cudaError_t e = cudaMemsetAsync(ctx.ws.keys, 0,
                                  sizeof(unsigned long long) * (size_t)a.gamma * ctx.cfg.R_max, s);
  if (e != cudaSuccess) return e;
  const int grid = simt_grid(ctx, a.V);
  if (a.cand_tok) {   // keep the Markov candidate lists of every step
    sp.cand = 1;
    sp.cand_parts = ctx.ws.cand_parts;
    sp.cand_R = ctx.cfg.R_max < kCandMaxR ? ctx.cfg.R_max : kCandMaxR;
  }
  if (a.gate_h) {   // gated or RNN head: the hidden-state parts of every position, once
    sp.A = a.gated_rep;
    e = a.rnn_W ? launch_rnn_h(ctx, a, s) : launch_gate_h(ctx, a, s);
    if (e != cudaSuccess) return e;
  }
  for (int j = 0; j < a.gamma; ++j) {
    sp.j = j;
    if (a.gate_h) {   // this step's representation from the tokens of the last
      e = a.rnn_W ? launch_rnn_step(ctx, a, j, s) : launch_gate_step(ctx, a, j, s);
      if (e != cudaSuccess) return e;
    }
    e = launch_simt(sp, ctx.cfg.dtype, grid, s, kModeStep);
    if (e != cudaSuccess) return e;
    count_launch(ctx);
  }
  return cudaSuccess;
}

cudaError_t launch_residual_simt(const Ctx& ctx, const VerifyArgs& a, cudaStream_t s) {
  SimtParams sp = base_params(ctx, a.R, a.V, a.rank, a.gamma, a.act, a.bias_at_first,
                              a.temperature, a.seed);
  sp.U = a.U;
  sp.E = a.E;
  sp.W = a.W;
  sp.P = a.P;
  sp.prev_tok = a.prev_tok;
  sp.tokens = a.tokens;
  sp.req_id = a.req_id;
  sp.lse_q = a.lse_q;
  sp.A = a.gated_rep;
  sp.keys = ctx.ws.res_keys;
  sp.res_sums = ctx.ws.res_sums;
  sp.rej_list = ctx.ws.rej_list;
  sp.rej_k = ctx.ws.rej_k;
  sp.rej_lseP = ctx.ws.rej_lseP;
  sp.n_rej = ctx.ws.counters + 1;
  count_launch(ctx);
  return launch_simt(sp, ctx.cfg.dtype, simt_grid(ctx, a.V), s, kModeResidual);
}

// ---------------------------------------------------------------------------
// Finalize: per (r, j) combine the CTA partials into lse_q, take the token
// from the argmax key and the (scaled) logit of the chosen token; per r the
// prefix survival in fp64 ("DSpark 论文精读" 3.1).
// ---------------------------------------------------------------------------
struct FinParams {
  const void* U;
  const void* E;
  const void* W;
  const float* conf;
  const int32_t* prev_tok;
  const float* A;                 // gated head representations, or nullptr
  const unsigned long long* keys;
  const float2* parts;
  int* status;
  int32_t* tokens;
  float* lse_q;
  float* logit_at_tok;
  float* survival;
  int R, R_max, V, rank, gamma, act, bias_at_first, n_part, n_used, sampled;
  float inv_T;
  int n_fin;            // CTAs of the finalize; any further CTAs run the schedule
  SchedParams sp;
};

template <typename T>
__global__ void __launch_bounds__(256) propose_finalize_kernel(FinParams p) {
  static_assert(kSchedThreads == 256, "schedule CTAs share the finalize's block size");
  if ((int)blockIdx.x >= p.n_fin) {
    extern __shared__ __align__(16) unsigned char sched_smem[];
    schedule_cta(p.sp, blockIdx.x - p.n_fin, gridDim.x - p.n_fin, sched_smem);
    return;
  }
  const int lane = threadIdx.x & 31;
  const int pair = blockIdx.x * 8 + (threadIdx.x >> 5);
  const T* U = static_cast<const T*>(p.U);
  const T* E = static_cast<const T*>(p.E);
  const T* W = static_cast<const T*>(p.W);

  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g < p.R) {
    double acc = 1.0;
    for (int j = 0; j < p.gamma; ++j) {
      float c = p.conf[(size_t)g * p.gamma + j];
      if (!isfinite(c)) {
        set_status(p.status, kErrNonfinite);
        c = 0.f;
      }
      c = fminf(fmaxf(c, 0.f), 1.f);
      acc *= (double)c;
      p.survival[(size_t)g * p.gamma + j] = (float)acc;
    }
  }
  if (pair >= p.R * p.gamma) return;
  const int r = pair / p.gamma, j = pair - r * p.gamma;
  Lse2 l = lse2_empty();
  for (int c = lane; c < p.n_used; c += 32) {
    const float2 q = p.parts[((size_t)j * p.n_part + c) * p.R_max + r];
    l = lse2_merge(l, Lse2{q.x, q.y});
  }
  l = warp_lse2(l);
  const unsigned long long key = p.keys[(size_t)j * p.R_max + r];
  const uint32_t x = key_index(key);
  const float lse = lse2_value(l);
  float logit;
  if (!p.sampled) {
    logit = key_value(key);
  } else {
    float dot = 0.f;
    if ((j > 0 || p.bias_at_first) && x < (uint32_t)p.V) {
      int prev = (j == 0) ? p.prev_tok[r] : (int)key_index(p.keys[(size_t)(j - 1) * p.R_max + r]);
      if (prev < 0 || prev >= p.V) prev = 0;
      const float* arow = p.A ? p.A + ((size_t)r * p.gamma + j) * p.rank : nullptr;
      for (int k = lane; k < p.rank; k += 32)
        dot = fmaf(arow ? arow[k] : act_apply(ld_elem(E, (size_t)prev * p.rank + k), p.act),
                   ld_elem(W, (size_t)x * p.rank + k), dot);
      dot = warp_sum(dot);
    }
    const float u = x < (uint32_t)p.V ? ld_elem(U, ((size_t)r * p.gamma + j) * p.V + x) : 0.f;
    logit = (u + dot) * p.inv_T;
  }
  if (lane == 0) {
    p.tokens[(size_t)r * p.gamma + j] = (int32_t)x;
    p.lse_q[(size_t)r * p.gamma + j] = lse;
    p.logit_at_tok[(size_t)r * p.gamma + j] = logit;
    if (!isfinite(lse) || !isfinite(logit) || key == 0ull) set_status(p.status, kErrNonfinite);
  }
}

cudaError_t launch_propose_finalize_n(const Ctx& ctx, const ProposeArgs& a, int n_used,
                                      cudaStream_t s) {
  FinParams p{};
  p.U = a.U;
  p.E = a.E;
  p.W = a.W;
  p.conf = a.conf;
  p.prev_tok = a.prev_tok;
  p.A = a.gate_h ? a.gated_rep : nullptr;
  p.keys = ctx.ws.keys;
  p.parts = ctx.ws.lse_parts;
  p.status = ctx.ws.status;
  p.tokens = a.tokens;
  p.lse_q = a.lse_q;
  p.logit_at_tok = a.logit_at_tok;
  p.survival = a.survival;
  p.R = a.R;
  p.R_max = ctx.cfg.R_max;
  p.V = a.V;
  p.rank = a.rank;
  p.gamma = a.gamma;
  p.act = a.act;
  p.bias_at_first = a.bias_at_first;
  p.n_part = ctx.n_part;
  p.n_used = n_used;
  p.sampled = a.temperature > 0.f ? 1 : 0;
  p.inv_T = a.temperature > 0.f ? 1.f / a.temperature : 1.f;
  const int pairs = a.R * a.gamma;
  int grid = (pairs + 7) / 8;
  const int gsurv = (a.R + 255) / 256;
  if (grid < gsurv) grid = gsurv;
  p.n_fin = grid;
  size_t smem = 0;
  if (a.sched_keep) {
    // the cycle's schedule in extra CTAs, from the confidences directly
    p.sp = make_sched_params(ctx, a.R, nullptr, a.conf, a.sched_sps, a.sched_n_sps, a.sched_keep,
                             a.sched_theta);
    grid += schedule_ctas(ctx, a.R);
    smem = schedule_smem_bytes(a.R, a.gamma);
  }
  if (ctx.cfg.dtype == 1) {
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(propose_finalize_kernel<__nv_bfloat16>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    propose_finalize_kernel<__nv_bfloat16><<<grid, 256, smem, s>>>(p);
  } else {
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(propose_finalize_kernel<float>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    propose_finalize_kernel<float><<<grid, 256, smem, s>>>(p);
  }
  count_launch(ctx);
  return cudaGetLastError();
}

cudaError_t launch_propose_finalize(const Ctx& ctx, const ProposeArgs& a, cudaStream_t s) {
  return launch_propose_finalize_n(ctx, a, simt_grid(ctx, a.V), s);
}

// ---------------------------------------------------------------------------
// Candidate sets: per (r, j) the top-kCandK of the CTAs' sorted lists.  Lane
// l of the row's warp owns lists l, l + 32, ... (at most kCandLPL); each of
// kCandK rounds takes the warp-wide maximum of the list heads and advances
// the list that held it.
// ---------------------------------------------------------------------------
constexpr int kCandLPL = 16;   // lists per lane: n_used <= 512

__global__ void __launch_bounds__(256) cand_finalize_kernel(const unsigned long long* parts,
                                                            int n_used, int n_part, int cand_R,
                                                            int R, int gamma, int32_t* tok,
                                                            float* logit) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= R * gamma) return;
  const int r = row / gamma, j = row - r * gamma;
  const unsigned long long* base = parts + (size_t)j * n_part * cand_R * kCandK;
  unsigned long long head[kCandLPL];
  int pos[kCandLPL];
#pragma unroll
  for (int i = 0; i < kCandLPL; ++i) {
    const int c = lane + 32 * i;
    pos[i] = 0;
    head[i] = c < n_used ? base[((size_t)c * cand_R + r) * kCandK] : 0ull;
  }
  for (int t = 0; t < kCandK; ++t) {
    unsigned long long lm = 0ull;
    int li = 0;
#pragma unroll
    for (int i = 0; i < kCandLPL; ++i)
      if (head[i] > lm) {
        lm = head[i];
        li = i;
      }
    const unsigned long long wm = warp_max_u64(lm);
    if (wm != 0ull && lm == wm) {
#pragma unroll
      for (int i = 0; i < kCandLPL; ++i)
        if (i == li) {
          ++pos[i];
          head[i] = pos[i] < kCandK
                        ? base[((size_t)(lane + 32 * i) * cand_R + r) * kCandK + pos[i]]
                        : 0ull;
        }
    }
    if (lane == 0) {
      tok[(size_t)row * kCandK + t] = wm ? (int32_t)key_index(wm) : -1;
      logit[(size_t)row * kCandK + t] = wm ? key_value(wm) : -INFINITY;
    }
  }
}

cudaError_t launch_cand_finalize(const Ctx& ctx, const ProposeArgs& a, int n_used, cudaStream_t s) {
  const int rows = a.R * a.gamma;
  const int cand_R = ctx.cfg.R_max < kCandMaxR ? ctx.cfg.R_max : kCandMaxR;
  cand_finalize_kernel<<<(rows + 7) / 8, 256, 0, s>>>(ctx.ws.cand_parts, n_used, ctx.n_part, cand_R,
                                                      a.R, a.gamma, a.cand_tok, a.cand_logit);
  count_launch(ctx);
  return cudaGetLastError();
}

}  // namespace dsd
