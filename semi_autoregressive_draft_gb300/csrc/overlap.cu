// Offline teacher-forced overlap metrics ("Qwen3.8-Flash-Next DSpark 训练实验",
// 评估口径 / 离线指标; "DSpark 论文精读" 3.1 overlap identity).
//
// Per valid (block n, position i): p = softmax(P[n,i]), q = softmax(Q[n,i]),
// a = sum_v min(p, q) and l1 = sum_v |p - q| = sum_v max(p, q) - min(p, q).
// Both need the two log-normalisers first, so every row is read twice (from
// shared memory in the split kernel).
//
// overlap_split: one cluster of eight CTAs per (n, i) pair, each CTA owning
// one eighth of the vocabulary.  Two 1-D bulk copies put the CTA's slices of
// the P and Q rows in shared memory (76 KB at V = 151,936 bf16, two CTAs per
// SM); pass 1 reduces them to base-2 log-sum-exp partials, which every CTA
// pushes into every peer's inbox with st.async (completing the peer's
// mbarrier); each CTA merges the eight partials in a fixed tree (the same
// normalisers, bit for bit, in every CTA); pass 2 sums min(p, q) =
// 2^min(log2 p, log2 q) from shared memory, one 2^x per position.  CTA 0
// collects the eight sums and writes a and l1 = sum p + sum q - 2 sum
// min(p, q).  Every byte crosses HBM once.  (Clusters of 16 CTAs with half
// the slice, four CTAs per SM, were measured slower: 3.95 against 3.51 ms
// on 4096 blocks.)
// overlap_rows (only when the split grid would exceed the launch limit): one
// CTA per pair, two passes over the rows.
// overlap_finalize: one CTA; tau per block, accept_rate per position over
// the valid blocks, mean tau over the valid blocks, all summed in a fixed
// order in fp64 so the result does not depend on scheduling.
#include "tc_common.cuh"

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

// ------------------------------------------------------------------------
// overlap_split
// ------------------------------------------------------------------------
constexpr int kOsCluster = 8;        // CTAs per row pair (portable cluster maximum)
constexpr int kOsThreads = 256;
constexpr int kOsWarps = kOsThreads / 32;
static_assert((kOsWarps & (kOsWarps - 1)) == 0 && kOsWarps <= 32, "warp tree over lanes");
static_assert((kOsCluster & (kOsCluster - 1)) == 0 && kOsCluster <= 32, "CTA tree over lanes");

namespace os {
// shared-memory address of the same variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(tc::smem_u32(p)), "r"(rank));
  return r;
}
// Asynchronous store into a peer CTA's shared memory that completes 16 (or 4)
// bytes of the transaction count of the peer's mbarrier `rbar`.
__device__ __forceinline__ void st_async_f4(uint32_t raddr, float4 v, uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
          raddr),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(rbar)
      : "memory");
}
__device__ __forceinline__ void st_async_f1(uint32_t raddr, float x, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(raddr),
               "f"(x), "r"(rbar)
               : "memory");
}
// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global memory into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(tc::smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(tc::smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t pack2u(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ float lo_f(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_f(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

// 16 bytes of logits as packed pairs of fp32 (bf16 -> fp32 is exact).
template <typename T>
constexpr int pairs_per_chunk() {
  return sizeof(T) == 2 ? 4 : 2;
}
template <typename T>
__device__ __forceinline__ void to_pairs(uint4 q, uint64_t (&x)[4]) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = pack2u(w[i] << 16, w[i] & 0xFFFF0000u);
  } else {
    x[0] = pack2u(q.x, q.y);
    x[1] = pack2u(q.z, q.w);
    x[2] = x[3] = 0ull;
  }
}
// The same vocabulary positions of both rows as packed (P, Q) pairs.
template <typename T>
__device__ __forceinline__ void cross_pairs(uint4 qp, uint4 qq, uint64_t (&e)[8]) {
  const uint32_t wp[4] = {qp.x, qp.y, qp.z, qp.w}, wq[4] = {qq.x, qq.y, qq.z, qq.w};
  if constexpr (sizeof(T) == 2) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      e[2 * i] = pack2u(wp[i] << 16, wq[i] << 16);
      e[2 * i + 1] = pack2u(wp[i] & 0xFFFF0000u, wq[i] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) e[i] = pack2u(wp[i], wq[i]);
    e[4] = e[5] = e[6] = e[7] = 0ull;
  }
}
template <typename T>
__device__ __forceinline__ float chunk_max(const uint64_t (&x)[4]) {
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < pairs_per_chunk<T>(); ++i) m = tc::max3(m, lo_f(x[i]), hi_f(x[i]));
  return m;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// Sum over this thread's chunks (c = tid, tid + kOsThreads, ...) of one row
// (in shared memory) of 2^(x log2e - ref).
template <typename T>
__device__ __forceinline__ float sum_exp(const unsigned char* row, int nchunks, int tid, float ref) {
  const uint64_t l2 = tc::pack2(kLog2e, kLog2e), nr = tc::pack2(-ref, -ref);
  uint64_t acc = 0ull;
  for (int c = tid; c < nchunks; c += kOsThreads) {
    uint64_t x[4];
    to_pairs<T>(*reinterpret_cast<const uint4*>(row + 16 * c), x);
#pragma unroll
    for (int i = 0; i < pairs_per_chunk<T>(); ++i) {
      const uint64_t d = tc::fma2(x[i], l2, nr);
      acc = tc::add2(acc, tc::pack2(tc::ex2(lo_f(d)), tc::ex2(hi_f(d))));
    }
  }
  return lo_f(acc) + hi_f(acc);
}
// The exact base-2 log-sum-exp state of one warp's chunks of one row (in
// shared memory): its maximum first, then the sum.  Every lane returns the
// warp's state.  The slow path of pass 1.
template <typename T>
__device__ Lse2 warp_exact_lse(const unsigned char* row, int nchunks, int tid) {
  float e = -INFINITY;
  for (int c = tid; c < nchunks; c += kOsThreads) {
    uint64_t x[4];
    to_pairs<T>(*reinterpret_cast<const uint4*>(row + 16 * c), x);
    e = fmaxf(e, chunk_max<T>(x));
  }
  const float m = warp_max(e) * kLog2e;
  if (m == -INFINITY) return lse2_empty();
  return Lse2{m, warp_sum(sum_exp<T>(row, nchunks, tid, m))};   // NaN / inf stay non-finite
}
// Pass 1 of one warp: the base-2 log-sum-exp states of its chunks of both
// rows (every lane returns the warp's states).  The reference of each row is
// the warp's maximum over its lanes' first chunks; a row whose later logits
// exceed it so far that a term overflows (or whose first chunks are all
// -inf) takes the exact path.
template <typename T>
__device__ __forceinline__ void warp_pass1(const unsigned char* pr, const unsigned char* qr,
                                           int nchunks, int tid, Lse2& wp, Lse2& wq) {
  const uint64_t l2 = tc::pack2(kLog2e, kLog2e);
  uint64_t x[4], y[4];
  float rp = -INFINITY, rq = -INFINITY;
  if (tid < nchunks) {
    to_pairs<T>(*reinterpret_cast<const uint4*>(pr + 16 * tid), x);
    to_pairs<T>(*reinterpret_cast<const uint4*>(qr + 16 * tid), y);
    rp = chunk_max<T>(x);
    rq = chunk_max<T>(y);
  }
  rp = warp_max(rp) * kLog2e;
  rq = warp_max(rq) * kLog2e;
  const uint64_t np = tc::pack2(-rp, -rp), nq = tc::pack2(-rq, -rq);
  uint64_t ap = 0ull, aq = 0ull;
  for (int c = tid; c < nchunks; c += kOsThreads) {
    if (c != tid) {
      to_pairs<T>(*reinterpret_cast<const uint4*>(pr + 16 * c), x);
      to_pairs<T>(*reinterpret_cast<const uint4*>(qr + 16 * c), y);
    }
#pragma unroll
    for (int i = 0; i < pairs_per_chunk<T>(); ++i) {
      const uint64_t d = tc::fma2(x[i], l2, np), e = tc::fma2(y[i], l2, nq);
      ap = tc::add2(ap, tc::pack2(tc::ex2(lo_f(d)), tc::ex2(hi_f(d))));
      aq = tc::add2(aq, tc::pack2(tc::ex2(lo_f(e)), tc::ex2(hi_f(e))));
    }
  }
  const float sp = warp_sum(lo_f(ap) + hi_f(ap)), sq = warp_sum(lo_f(aq) + hi_f(aq));
  // the tests below are uniform across the warp
  wp = (rp == -INFINITY || !(sp <= 3.0e38f)) ? warp_exact_lse<T>(pr, nchunks, tid) : Lse2{rp, sp};
  wq = (rq == -INFINITY || !(sq <= 3.0e38f)) ? warp_exact_lse<T>(qr, nchunks, tid) : Lse2{rq, sq};
}
// Merge of two base-2 states with the special-function unit's 2^x.
__device__ __forceinline__ Lse2 merge_fast(Lse2 a, Lse2 b) {
  const float M = fmaxf(a.m, b.m);
  if (M == -INFINITY) return lse2_empty();
  return Lse2{M, fmaf(a.s, tc::ex2(a.m - M), b.s * tc::ex2(b.m - M))};
}
// Sum of min(p, q) over this thread's chunks, with nlp = -log2 normaliser of
// P and nlq = -log2 normaliser of Q (both splat to pairs): two adjacent
// positions per packed operation, one 2^x per position.
template <typename T>
__device__ __forceinline__ float slice_summin(const unsigned char* pr, const unsigned char* qr,
                                              int nchunks, int tid, uint64_t nlp, uint64_t nlq) {
  const uint64_t l2 = tc::pack2(kLog2e, kLog2e);
  uint64_t acc = 0ull;
  for (int c = tid; c < nchunks; c += kOsThreads) {
    uint64_t x[4], y[4];
    to_pairs<T>(*reinterpret_cast<const uint4*>(pr + 16 * c), x);
    to_pairs<T>(*reinterpret_cast<const uint4*>(qr + 16 * c), y);
#pragma unroll
    for (int i = 0; i < pairs_per_chunk<T>(); ++i) {
      const uint64_t dp = tc::fma2(x[i], l2, nlp), dq = tc::fma2(y[i], l2, nlq);   // log2 p, log2 q
      acc = tc::add2(acc, tc::pack2(tc::ex2(fminf(lo_f(dp), lo_f(dq))),
                                    tc::ex2(fminf(hi_f(dp), hi_f(dq)))));
    }
  }
  return lo_f(acc) + hi_f(acc);
}
}  // namespace os


struct OsParams {
  const unsigned char* P;   // [N * gamma][V] logits of type T
  const unsigned char* Q;
  const int32_t* valid_len;
  float* a_out;
  float* l1_out;
  int* status;
  long long row_bytes;      // V * sizeof(T), a multiple of 16
  int slice_bytes;          // vocabulary bytes per CTA, a multiple of 16
  int gamma;
};

// Bounded wait by one warp (lane 0 polls) on a barrier completed by copies
// or by peers' st.async; acquire at cluster scope so that peers' data is
// visible.
__device__ __forceinline__ void os_warp_wait(uint64_t* bar, volatile int* abort_flag, int* status) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) {
    ok = 0;
    for (uint32_t i = 0; i < kSpinLimit && !ok; ++i) {
      uint32_t r;
      asm volatile(
          "{\n\t.reg .pred p;\n\t"
          "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], 0;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(r)
          : "r"(tc::smem_u32(bar))
          : "memory");
      ok = (int)r;
      if (!ok && (i & 255u) == 255u && *abort_flag) break;
    }
    if (!ok) {
      set_status(status, kErrTimeout);
      *abort_flag = 1;
    }
  }
  __syncwarp();
}

template <typename T>
__global__ void __launch_bounds__(kOsThreads) overlap_split(OsParams p) {
  extern __shared__ __align__(128) unsigned char os_smem[];   // [P slice | Q slice]
  __shared__ __align__(8) uint64_t bar_data;   // the two slice copies
  __shared__ __align__(8) uint64_t bar_xch;    // the eight CTAs' partials (pushed by each)
  __shared__ __align__(8) uint64_t bar_sum;    // CTA 0: the eight CTAs' sums
  __shared__ __align__(16) float4 inbox[kOsCluster];   // (mP, sP, mQ, sQ) of every CTA
  __shared__ __align__(16) float sums[kOsCluster];     // CTA 0: every CTA's sum of min(p, q)
  __shared__ Lse2 red_p[kOsWarps], red_q[kOsWarps];
  __shared__ float red_s[kOsWarps];
  __shared__ float s_norm[2];
  __shared__ int s_abort;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = tc::cluster_ctarank();
  const int t = (int)(blockIdx.x / kOsCluster);   // the (block, position) pair
  const int n = t / p.gamma, i = t - n * p.gamma;
  int vl = __ldg(p.valid_len + n);
  if (vl < 0 || vl > p.gamma) {
    if (rank == 0 && tid == 0) set_status(p.status, kErrArg);
    vl = vl < 0 ? 0 : p.gamma;
  }
  if (i >= vl) {   // every CTA of the cluster leaves here, before any exchange
    if (rank == 0 && tid == 0) {
      p.a_out[t] = 0.f;
      p.l1_out[t] = 0.f;
    }
    return;
  }
  // this CTA's slice of both rows: bytes [lo, lo + len), copied to shared memory
  const int lo = (int)rank * p.slice_bytes;
  const long long rest = p.row_bytes - lo;
  const int len = rest <= 0 ? 0 : (rest < p.slice_bytes ? (int)rest : p.slice_bytes);
  const int nchunks = len >> 4;
  unsigned char* sp_row = os_smem;
  unsigned char* sq_row = os_smem + p.slice_bytes;
  if (tid == 0) {
    tc::mbar_init(&bar_data, 1);
    tc::mbar_init(&bar_xch, 1);
    tc::mbar_init(&bar_sum, 1);
    tc::mbar_fence_init();
    s_abort = 0;
    tc::mbar_arrive_expect_tx(&bar_data, 2u * (uint32_t)len);
    if (len > 0) {
      const size_t off = (size_t)t * (size_t)p.row_bytes + (size_t)lo;
      const uint64_t pol = policy_evict_first();
      os::bulk_load(sp_row, p.P + off, (uint32_t)len, &bar_data, pol);
      os::bulk_load(sq_row, p.Q + off, (uint32_t)len, &bar_data, pol);
    }
    // the peers' pushes complete these barriers' transactions
    tc::mbar_arrive_expect_tx(&bar_xch, (uint32_t)(kOsCluster * sizeof(float4)));
    if (rank == 0) tc::mbar_arrive_expect_tx(&bar_sum, (uint32_t)(kOsCluster * sizeof(float)));
  }
  // Barriers initialised cluster-wide before any peer pushes to them: arrive
  // now (thread 0's fence.mbarrier_init already released the initialisation
  // at cluster scope), wait just before the first push (by then every CTA
  // has arrived).
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  if (warp == 0) os_warp_wait(&bar_data, &s_abort, p.status);
  __syncthreads();
  // If a wait gave up (DSD_ERR_TIMEOUT is set), the sums below are
  // meaningless but every access stays in bounds.

  // pass 1: the slice's base-2 log-sum-exp partials of both rows
  Lse2 wp, wq;
  os::warp_pass1<T>(sp_row, sq_row, nchunks, tid, wp, wq);
  if (lane == 0) {
    red_p[warp] = wp;
    red_q[warp] = wq;
  }
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    // lane r < 8 pushes this CTA's partials into CTA r's inbox slot [rank]
    Lse2 lp = lse2_empty(), lq = lse2_empty();
    if (lane < kOsWarps) {
      lp = red_p[lane];
      lq = red_q[lane];
    }
#pragma unroll
    for (int o = 1; o < kOsWarps; o <<= 1) {
      lp = os::merge_fast(lp, Lse2{__shfl_xor_sync(0xffffffffu, lp.m, o),
                                   __shfl_xor_sync(0xffffffffu, lp.s, o)});
      lq = os::merge_fast(lq, Lse2{__shfl_xor_sync(0xffffffffu, lq.m, o),
                                   __shfl_xor_sync(0xffffffffu, lq.s, o)});
    }
    lp = Lse2{__shfl_sync(0xffffffffu, lp.m, 0), __shfl_sync(0xffffffffu, lp.s, 0)};
    lq = Lse2{__shfl_sync(0xffffffffu, lq.m, 0), __shfl_sync(0xffffffffu, lq.s, 0)};
    if (lane < kOsCluster)
      os::st_async_f4(os::peer_addr(&inbox[rank], (uint32_t)lane), make_float4(lp.m, lp.s, lq.m, lq.s),
                      os::peer_addr(&bar_xch, (uint32_t)lane));
    os_warp_wait(&bar_xch, &s_abort, p.status);
    // merge the eight slices in a fixed tree: the same bits in every CTA
    Lse2 mp = lse2_empty(), mq = lse2_empty();
    if (lane < kOsCluster) {
      const float4 v = inbox[lane];
      mp = Lse2{v.x, v.y};
      mq = Lse2{v.z, v.w};
    }
#pragma unroll
    for (int o = 1; o < kOsCluster; o <<= 1) {
      mp = os::merge_fast(mp, Lse2{__shfl_xor_sync(0xffffffffu, mp.m, o),
                                   __shfl_xor_sync(0xffffffffu, mp.s, o)});
      mq = os::merge_fast(mq, Lse2{__shfl_xor_sync(0xffffffffu, mq.m, o),
                                   __shfl_xor_sync(0xffffffffu, mq.s, o)});
    }
    if (lane == 0) {
      const float LP = mp.m + log2f(mp.s), LQ = mq.m + log2f(mq.s);
      if (rank == 0 && !(isfinite(LP) && isfinite(LQ))) set_status(p.status, kErrNonfinite);
      s_norm[0] = LP;
      s_norm[1] = LQ;
    }
  }
  __syncthreads();

  // pass 2: the slice's sum of min(p, q)
  const float nlp = -s_norm[0], nlq = -s_norm[1];
  float smin = os::slice_summin<T>(sp_row, sq_row, nchunks, tid, tc::pack2(nlp, nlp),
                                   tc::pack2(nlq, nlq));
  smin = warp_sum(smin);
  if (lane == 0) red_s[warp] = smin;
  __syncthreads();
  if (warp == 0) {
    if (lane == 0) {
      float v = 0.f;
      for (int w = 0; w < kOsWarps; ++w) v += red_s[w];
      os::st_async_f1(os::peer_addr(&sums[rank], 0u), v, os::peer_addr(&bar_sum, 0u));
    }
    if (rank == 0) {
      // CTA 0 stays until every CTA's sum has landed in its shared memory;
      // the other CTAs may leave: every push to them has already landed.
      // With p + q - |p - q| = 2 min(p, q) at every position,
      //   l1 = sum p + sum q - 2 sum min(p, q),
      // where sum p = sum_k s_k 2^(m_k - LP) over the slices' pass-1 partials
      // (1 up to rounding): the identity a = 1 - l1 / 2 then checks that the
      // two normalisers are consistent with the partials they came from.
      os_warp_wait(&bar_sum, &s_abort, p.status);
      float sp = 0.f, sq = 0.f;
      if (lane < kOsCluster) {
        const float4 v = inbox[lane];
        sp = v.y * tc::ex2(v.x - s_norm[0]);
        sq = v.w * tc::ex2(v.z - s_norm[1]);
        if (v.y == 0.f) sp = 0.f;   // an empty slice (m = -inf)
        if (v.w == 0.f) sq = 0.f;
      }
      sp = warp_sum(sp);
      sq = warp_sum(sq);
      if (lane == 0) {
        float a = 0.f;
        for (int r = 0; r < kOsCluster; ++r) a += sums[r];
        p.a_out[t] = a;
        p.l1_out[t] = sp + sq - 2.f * a;
      }
    }
  }
  if (tid == 0 && s_abort) drain_bar(&bar_data, 0u);   // no copy lands after the CTA is gone
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


// One cluster of kOsCluster CTAs per (block, position) pair; *done = false
// when the grid would exceed the launch limit or a slice pair would not fit
// in shared memory (V above about 900,000 bf16); the one-CTA-per-pair kernel
// then runs.
template <typename T>
cudaError_t launch_overlap_split(const Ctx& ctx, const OverlapArgs& a, cudaStream_t s, bool* done) {
  *done = false;
  const long long pairs = (long long)a.N * a.gamma;
  if (pairs * kOsCluster > 0x7fffffffLL) return cudaSuccess;
  const long long row_bytes = (long long)a.V * (long long)sizeof(T);
  OsParams p{};
  p.P = static_cast<const unsigned char*>(a.P);
  p.Q = static_cast<const unsigned char*>(a.Q);
  p.valid_len = a.valid_len;
  p.a_out = a.a;
  p.l1_out = a.l1;
  p.status = ctx.ws.status;
  p.row_bytes = row_bytes;
  p.slice_bytes = (int)(((row_bytes + kOsCluster - 1) / kOsCluster + 15) / 16 * 16);
  p.gamma = a.gamma;
  const int dyn = 2 * p.slice_bytes;
  int optin = 0, dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (dyn + 1024 > optin) return cudaSuccess;   // the two slices do not fit: fall back
  e = cudaFuncSetAttribute(overlap_split<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kOsCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pairs * kOsCluster));
  cfg.blockDim = dim3(kOsThreads);
  cfg.dynamicSmemBytes = (size_t)dyn;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, overlap_split<T>, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  count_launch(ctx);
  *done = true;
  return cudaSuccess;
}

cudaError_t launch_overlap(const Ctx& ctx, const OverlapArgs& a, cudaStream_t s) {
  if (a.N > 0) {
    bool done = false;
    cudaError_t e = a.dtype == 1
                        ? launch_overlap_split<__nv_bfloat16>(ctx, a, s, &done)
                        : launch_overlap_split<float>(ctx, a, s, &done);
    if (e != cudaSuccess) return e;
    if (!done) {
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
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  overlap_finalize<<<1, 1024, 0, s>>>(a.a, a.valid_len, a.N, a.gamma, a.tau, a.accept_rate,
                                      a.mean_tau);
  count_launch(ctx);
  return cudaGetLastError();
}

}  // namespace dsd
