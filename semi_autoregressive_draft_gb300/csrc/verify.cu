// Target-side rejection verification of the kept draft prefixes
// ("DeepSpec 训练全流程详解（以 Qwen3 + DSpark 为例）" 4.4 Verify;
// "DSpark 论文精读" 2.1 and 3.1).
//
// Kernels, in stream order:
//   verify_rows        persistent grid over (row, vocabulary split) items.
//                      Every CTA first scans keep_len + 1 into the row
//                      offsets in shared memory (row b belongs to the request
//                      whose offset range holds it), then streams only the B
//                      kept rows of P once (16-byte loads, evict-first),
//                      producing per split the base-2 lse of P/T and an
//                      argmax key (greedy: argmax P; sampled: the stream-3
//                      Gumbel-max of the bonus row).  The last CTA to finish
//                      (a ticket) decides every request, one thread each:
//                      it merges the splits, runs the accept tests in order
//                      and stops at the first rejection; writes accept_len
//                      and (unless a residual draw is needed) next_token.
//   residual pass      sampled only, requests with a rejection: recompute
//                      q_k from U, E, W (residual_tc_kernel on the tensor
//                      cores where the propose engine could run, else the
//                      CUDA-core bias path) and draw from
//                      norm(max(0, p_k - q_k)) by Gumbel-max (stream 2).
//   verify_finish      next_token of the rejected requests.
#include "dsd_common.cuh"

namespace dsd {

cudaError_t launch_residual_simt(const Ctx& ctx, const VerifyArgs& a, cudaStream_t s);
cudaError_t launch_residual_tc(const Ctx& ctx, const VerifyArgs& a, cudaStream_t s);
int tc_supported(const Ctx& ctx, char* why, size_t why_len);

// The residual pass runs on the tensor cores (residual_tc_kernel) wherever
// the propose engine could: bf16 tables, no activation, a rank that is a
// multiple of 64 (<= 256), the AUTO or TCGEN05 engine and the plain Markov
// head.  Otherwise the CUDA-core residual pass.
static bool residual_on_tc(const Ctx& ctx, const VerifyArgs& a) {
  if (a.gated_rep != nullptr || ctx.cfg.act != kActNone) return false;   // E rows as stored
  if (ctx.cfg.engine != 0 && ctx.cfg.engine != 2) return false;   // AUTO, TCGEN05
  char why[256];
  return tc_supported(ctx, why, sizeof(why)) != 0;
}

constexpr int kRowThreads = 256;
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

struct RowsParams {
  int* status;
  const void* P;
  const int32_t* keep_len;
  const uint32_t* req_id;
  RowPart* parts;
  unsigned int* ticket;     // CTAs finished, zero between calls
  // the decision
  const int32_t* tokens;
  const float* lse_q;
  const float* logit_at_tok;
  int32_t* accept_len;
  int32_t* next_token;
  int* rej_list;
  int* rej_k;
  float* rej_lseP;
  unsigned int* n_rej;
  int R, V, gamma, sampled;
  float inv_T;
  uint32_t k0, k1;
};

// One thread decides request r, whose rows start at item row `off` and
// whose kept prefix has L tokens: merge the splits of each row, run the
// accept tests in order, stop at the first rejection.  The parts were
// written by other CTAs before their ticket, so they are read from L2.
template <typename T>
__device__ void decide_request(const RowsParams& p, int r, int off, int L, int splits,
                               int splits_bonus) {
  const T* P = static_cast<const T*>(p.P);
  const uint32_t rid = p.req_id ? p.req_id[r] : (uint32_t)r;
  int k = L;
  float lseP_k = 0.f;
  unsigned long long key_k = 0ull;   // merged argmax key of row k, when known
  for (int t = 0; t < L; ++t) {
    const RowPart* rp = p.parts + (size_t)(off + t) * kVerifySplits;
    int x = p.tokens[(size_t)r * p.gamma + t];
    bool ok;
    if (!p.sampled) {
      unsigned long long key = 0ull;
#pragma unroll
      for (int q = 0; q < kVerifySplits; ++q)
        if (q < splits) {
          const unsigned long long kq = __ldcg(&rp[q].key);
          key = kq > key ? kq : key;
        }
      ok = (int)key_index(key) == x;
      key_k = key;
    } else {
      Lse2 l = lse2_empty();
#pragma unroll
      for (int q = 0; q < kVerifySplits; ++q)
        if (q < splits) {
          const float2 ms = __ldcg(reinterpret_cast<const float2*>(rp + q));
          l = lse2_merge(l, Lse2{ms.x, ms.y});
        }
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
    // greedy correction (row k rejected its token) or the bonus row L
    unsigned long long key = key_k;
    if (k == L) {
      const RowPart* rp = p.parts + (size_t)(off + L) * kVerifySplits;
      key = 0ull;
#pragma unroll
      for (int q = 0; q < kVerifySplits; ++q)
        if (q < splits_bonus) {
          const unsigned long long kq = __ldcg(&rp[q].key);
          key = kq > key ? kq : key;
        }
    }
    next = (int)key_index(key);
    if (key == 0ull) set_status(p.status, kErrNonfinite);
  } else {
    const unsigned int slot = atomicAdd(p.n_rej, 1u);
    p.rej_list[slot] = r;
    p.rej_k[r] = k;
    p.rej_lseP[r] = lseP_k;
  }
  p.accept_len[r] = k;
  p.next_token[r] = next;
}

// Per-thread state of one item: the online log-sum-exp of P/T (sampled), the
// Gumbel-max key of a bonus row (sampled), or the running maximum and its
// lowest index (greedy).
struct RowFold {
  Lse2 st;
  unsigned long long best;
  float bz;
  uint32_t bv;
  bool nan_seen;
};

__device__ __forceinline__ RowFold rowfold_empty() {
  RowFold f;
  f.st = lse2_empty();
  f.best = 0ull;
  f.bz = -INFINITY;
  f.bv = 0xFFFFFFFFu;
  f.nan_seen = false;
  return f;
}

// Fold one 16-byte vector of row t (vocabulary positions v0 ..) into f.
// Greedy: a vector's index is looked up only when its maximum beats the
// running one; NaN propagates through max.NaN and is reported.
template <typename T, bool SAMPLED>
__device__ __forceinline__ void fold_vec(RowFold& f, uint4 q, int v0, bool bonus, uint32_t t,
                                         uint32_t rid, const RowsParams& p) {
  constexpr int epc = 16 / (int)sizeof(T);
  if constexpr (!SAMPLED && sizeof(T) == 2) {
    // greedy bf16: the vector's maximum by packed bf16x2 maxima (exact); the
    // elements are unpacked only when it beats the running maximum
    const uint32_t m2 = bf16x2_max_nan(bf16x2_max_nan(q.x, q.y), bf16x2_max_nan(q.z, q.w));
    const float m = max_nan(bf16lo(m2), bf16hi(m2));
    if (!(m <= f.bz)) {          // a larger maximum, or NaN
      if (m != m) {
        f.nan_seen = true;
      } else {
        const float x[8] = {bf16lo(q.x), bf16hi(q.x), bf16lo(q.y), bf16hi(q.y),
                            bf16lo(q.z), bf16hi(q.z), bf16lo(q.w), bf16hi(q.w)};
        int idx = 7;
#pragma unroll
        for (int e = 6; e >= 0; --e)
          if (x[e] == m) idx = e;
        f.bz = m;
        f.bv = (uint32_t)(v0 + idx);
      }
    }
    return;
  }
  float x[8];
  if constexpr (sizeof(T) == 2) {
    x[0] = bf16lo(q.x); x[1] = bf16hi(q.x); x[2] = bf16lo(q.y); x[3] = bf16hi(q.y);
    x[4] = bf16lo(q.z); x[5] = bf16hi(q.z); x[6] = bf16lo(q.w); x[7] = bf16hi(q.w);
  } else {
    x[0] = __uint_as_float(q.x); x[1] = __uint_as_float(q.y);
    x[2] = __uint_as_float(q.z); x[3] = __uint_as_float(q.w);
  }
  if constexpr (!SAMPLED) {
    float m = max3_nan(x[0], x[1], x[2]);
#pragma unroll
    for (int e = 3; e < epc; e += 2)
      m = e + 1 < epc ? max3_nan(m, x[e], x[e + 1]) : max_nan(m, x[e]);
    if (!(m <= f.bz)) {          // a larger maximum, or NaN
      if (m != m) {
        f.nan_seen = true;
      } else {
        int idx = epc - 1;
#pragma unroll
        for (int e = epc - 2; e >= 0; --e)
          if (x[e] == m) idx = e;
        f.bz = m;
        f.bv = (uint32_t)(v0 + idx);
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < epc; ++e) x[e] *= p.inv_T;
    if (!bonus) {
      // a tested row: the normaliser of P/T (a bonus row needs only its key)
      float cmax = -INFINITY;
#pragma unroll
      for (int e = 0; e < epc; ++e) cmax = fmaxf(cmax, x[e] * kLog2e);
      const float M = fmaxf(f.st.m, cmax);
      float s = f.st.s * exp2f(f.st.m - M);
#pragma unroll
      for (int e = 0; e < epc; ++e) s += exp2f(fmaf(x[e], kLog2e, -M));
      f.st.m = M;
      f.st.s = s;
    } else {
      // a bonus row: the Gumbel-max draw as a running (value, index) pair,
      // the first maximum kept (a later entry must be strictly larger; a
      // NaN logit never wins)
#pragma unroll
      for (int e = 0; e < epc; e += 4) {
        const uint32_t v = (uint32_t)(v0 + e);
        const Philox4 ph = philox4x32_10(v >> 2, t, rid, 3u, p.k0, p.k1);
        // v0 is a multiple of 4 (epc-aligned), so words map to v .. v+3
        const float z0 = x[e + 0] + gumbel_from_word(ph.x);
        const float z1 = x[e + 1] + gumbel_from_word(ph.y);
        const float z2 = x[e + 2] + gumbel_from_word(ph.z);
        const float z3 = x[e + 3] + gumbel_from_word(ph.w);
        if (z0 > f.bz) { f.bz = z0; f.bv = v + 0; }
        if (z1 > f.bz) { f.bz = z1; f.bv = v + 1; }
        if (z2 > f.bz) { f.bz = z2; f.bv = v + 2; }
        if (z3 > f.bz) { f.bz = z3; f.bv = v + 3; }
      }
    }
  }
}

// Shared memory of the row pass besides the ring: the row offsets and the
// block reduction.
struct RowsShared {
  Lse2 red_l[kRowThreads / 32];
  unsigned long long red_k[kRowThreads / 32];
  int scan_w[kRowThreads / 32];
  int last;
};

// Row offsets: exclusive scan of clamp(keep_len) + 1 into s_off[0..R], with
// s_off[R] = B.  Row b belongs to the request r with s_off[r] <= b <
// s_off[r + 1].
__device__ __forceinline__ void row_offsets(const RowsParams& p, int* s_off, RowsShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int IPT = (p.R + kRowThreads - 1) / kRowThreads;
  const int r0 = tid * IPT;
  int local = 0;
  for (int q = 0; q < IPT; ++q) {
    const int r = r0 + q;
    if (r < p.R) {
      int L = p.keep_len[r];
      if (L < 0 || L > p.gamma) {
        if (blockIdx.x == 0) set_status(p.status, kErrArg);
        L = L < 0 ? 0 : p.gamma;
      }
      s_off[r] = L + 1;          // the row count, turned into an offset below
      local += L + 1;
    }
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh.scan_w[warp] = incl;
  __syncthreads();
  int wbase = 0;
  for (int w = 0; w < warp; ++w) wbase += sh.scan_w[w];
  int off = wbase + incl - local;
  for (int q = 0; q < IPT; ++q) {
    const int r = r0 + q;
    if (r < p.R) {
      const int n = s_off[r];
      s_off[r] = off;
      off += n;
    }
  }
  if (tid == kRowThreads - 1) s_off[p.R] = off;   // the last thread ends at B
  __syncthreads();
}

// The request of row b: the largest r with s_off[r] <= b.
__device__ __forceinline__ int row_request(const int* s_off, int R, int b) {
  int lo = 0, hi = R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_off[mid] <= b)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Block reduction of one item's folds; thread 0 writes the item's part.
template <bool SAMPLED>
__device__ __forceinline__ void finish_item(const RowsParams& p, RowFold& f, int part, int v_first,
                                            int v_end, bool bonus, RowsShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // greedy rows and sampled bonus rows: the thread's (value, index) pair
  // as a packed key (tested rows of the sampled path keep no key)
  if ((!SAMPLED || bonus) && v_first < v_end) {
    if (f.nan_seen) set_status(p.status, kErrNonfinite);
    // every element was -inf: the first one holds the maximum
    f.best = make_key(f.bz, f.bv == 0xFFFFFFFFu ? (uint32_t)v_first : f.bv);
  }
  if constexpr (SAMPLED) f.st = warp_lse2(f.st);   // greedy rows have no normaliser
  f.best = warp_max_u64(f.best);
  if (lane == 0) {
    sh.red_l[warp] = f.st;
    sh.red_k[warp] = f.best;
  }
  __syncthreads();
  if (tid == 0) {
    Lse2 l = lse2_empty();
    unsigned long long k = 0ull;
    for (int w = 0; w < kRowThreads / 32; ++w) {
      if constexpr (SAMPLED) l = lse2_merge(l, sh.red_l[w]);
      k = sh.red_k[w] > k ? sh.red_k[w] : k;
    }
    p.parts[part] = RowPart{l.m, l.s, k};
  }
  __syncthreads();
}

// The last CTA to finish (a ticket) decides every request, one thread each.
template <typename T>
__device__ __forceinline__ void decide_all(const RowsParams& p, const int* s_off, int splits,
                                           int splits_bonus, RowsShared& sh) {
  const int tid = threadIdx.x;
  __threadfence();
  __syncthreads();
  if (tid == 0) sh.last = (atomicAdd(p.ticket, 1u) == gridDim.x - 1) ? 1 : 0;
  __syncthreads();
  if (!sh.last) return;
  __threadfence();
  for (int r = tid; r < p.R; r += kRowThreads)
    decide_request<T>(p, r, s_off[r], s_off[r + 1] - s_off[r] - 1, splits, splits_bonus);
  if (tid == 0) *p.ticket = 0u;   // ready for the next call on the stream
}

// Plain-load row pass, for P in host memory read in place (or a ring that
// does not fit): items are spread over a persistent grid, several 16-byte
// loads in flight per thread (eight for greedy rows, four with the sampled
// path's larger register set).
template <typename T, bool SAMPLED>
__global__ void __launch_bounds__(kRowThreads, 4) verify_rows(RowsParams p) {
  constexpr int epc = 16 / (int)sizeof(T);
  extern __shared__ int s_off[];   // [R + 1]
  __shared__ RowsShared sh;
  row_offsets(p, s_off, sh);
  // Rows are split into as many vocabulary chunks as keep every CTA busy
  // with about one item (at most kVerifySplits): fewer, longer items stream
  // more bytes per block reduction.  Greedy rows all cost the same.  In the
  // sampled path a bonus row also draws a Philox-Gumbel key per entry, about
  // four times a tested row's work, so bonus rows get four times the splits
  // and the items cost about the same: the tested rows' items come first,
  // then the bonus rows'.
  const int B = s_off[p.R];
  int splits, splits_bonus;
  if (!SAMPLED) {
    splits = splits_bonus = max(1, min(kVerifySplits, (int)gridDim.x / B));
  } else {
    const int n_tested = B - p.R;
    splits = max(1, min(kVerifySplits / 4, (int)gridDim.x / (n_tested + 4 * p.R)));
    splits_bonus = 4 * splits;
  }
  const int chunk = ((p.V + splits - 1) / splits + epc - 1) / epc * epc;
  const int chunk_bonus = ((p.V + splits_bonus - 1) / splits_bonus + epc - 1) / epc * epc;
  const int n_tested_items = SAMPLED ? (B - p.R) * splits : 0;
  const int n_items = SAMPLED ? n_tested_items + p.R * splits_bonus : B * splits;
  const T* P = static_cast<const T*>(p.P);
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    int r, t, sp, ck;
    if (!SAMPLED) {
      const int b = item / splits;
      sp = item - b * splits;
      r = row_request(s_off, p.R, b);
      t = b - s_off[r];
      ck = chunk;
    } else if (item < n_tested_items) {
      // k-th tested row: request r holds tested rows s_off[r] - r ..
      // s_off[r + 1] - r - 2 of the tested order
      const int k = item / splits;
      sp = item - k * splits;
      int lo = 0, hi = p.R - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_off[mid] - mid <= k)
          lo = mid;
        else
          hi = mid - 1;
      }
      r = lo;
      t = k - (s_off[r] - r);
      ck = chunk;
    } else {
      const int q = item - n_tested_items;
      r = q / splits_bonus;
      sp = q - r * splits_bonus;
      t = s_off[r + 1] - s_off[r] - 1;
      ck = chunk_bonus;
    }
    const int b = s_off[r] + t;
    const bool bonus = (t == s_off[r + 1] - s_off[r] - 1);
    const uint32_t rid = p.req_id ? p.req_id[r] : (uint32_t)r;
    const T* row = P + ((size_t)r * (p.gamma + 1) + t) * p.V;
    const int v_begin = sp * ck;
    const int v_end = min(p.V, v_begin + ck);
    const int v_first = v_begin + (int)threadIdx.x * epc;
    RowFold f = rowfold_empty();
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
        fold_vec<T, SAMPLED>(f, q[u], v0, bonus, (uint32_t)t, rid, p);
      }
    }
    finish_item<SAMPLED>(p, f, b * kVerifySplits + sp, v_first, v_end, bonus, sh);
  }
  decide_all<T>(p, s_off, splits, splits_bonus, sh);
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
  cudaError_t e;
  if (sampled) {
    e = cudaMemsetAsync(ws.counters, 0, 16 * sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(ws.res_keys, 0, 2 * sizeof(unsigned long long) * ctx.cfg.R_max, s);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(ws.res_sums, 0, 2 * sizeof(float) * ctx.cfg.R_max, s);
    if (e != cudaSuccess) return e;
  }

  RowsParams rp{};
  rp.status = ws.status;
  rp.P = a.P;
  rp.keep_len = a.keep_len;
  rp.req_id = a.req_id;
  rp.parts = ws.vparts;
  rp.ticket = ws.tickets + 3;
  rp.tokens = a.tokens;
  rp.lse_q = a.lse_q;
  rp.logit_at_tok = a.logit_at_tok;
  rp.accept_len = a.accept_len;
  rp.next_token = a.next_token;
  rp.rej_list = ws.rej_list;
  rp.rej_k = ws.rej_k;
  rp.rej_lseP = ws.rej_lseP;
  rp.n_rej = ws.counters + 1;
  rp.R = a.R;
  rp.V = a.V;
  rp.gamma = a.gamma;
  rp.sampled = sampled;
  rp.inv_T = inv_T;
  rp.k0 = k0;
  rp.k1 = k1;
  const int grid_rows = ctx.num_sms * 4;
  const size_t smem = (size_t)(a.R + 1) * sizeof(int);
  if (ctx.cfg.dtype == 1) {
    if (sampled)
      verify_rows<__nv_bfloat16, true><<<grid_rows, kRowThreads, smem, s>>>(rp);
    else
      verify_rows<__nv_bfloat16, false><<<grid_rows, kRowThreads, smem, s>>>(rp);
  } else {
    if (sampled)
      verify_rows<float, true><<<grid_rows, kRowThreads, smem, s>>>(rp);
    else
      verify_rows<float, false><<<grid_rows, kRowThreads, smem, s>>>(rp);
  }
  count_launch(ctx);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  if (sampled) {
    e = residual_on_tc(ctx, a) ? launch_residual_tc(ctx, a, s) : launch_residual_simt(ctx, a, s);
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
