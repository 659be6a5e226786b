// Per-step work of the sequential heads that read the backbone's hidden
// state ("DSpark 论文精读" 2.3, GatedMarkovHead and RNNHead; "DSpark notes"
// 2.3), one output per warp.  The standalone step kernels (gated.cu) and the
// single-launch tensor-core propose kernel (propose_tc.cu) both call these,
// so the two paths compute every representation with the same arithmetic in
// the same order.
//
// Gated head:  m = act(E[x_{j-1}]),  g = sigmoid(W_g [h_j; m]),  a = g * m.
// RNN head:    u = [s_{j-1}; m; h_j],  g = sigmoid(W_g u),  c = tanh(W_c u),
//              s_j = g * s_{j-1} + (1 - g) * c,  a = tanh(W_o [s_j; m; h_j]).
// The hidden-state parts (W h_j) come precomputed as split-K partials Zh,
// added in split order.  Values written earlier in the same launch (the
// draft keys, the RNN state) are read through L2 (ld.global.cg).
#pragma once

#include "dsd_common.cuh"

namespace dsd {

// Eight consecutive elements of a weight row (16-byte aligned), as fp32.
template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&x)[8]) {
  const uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
  if constexpr (sizeof(T) == 2) {
    x[0] = bf16lo(q.x); x[1] = bf16hi(q.x); x[2] = bf16lo(q.y); x[3] = bf16hi(q.y);
    x[4] = bf16lo(q.z); x[5] = bf16hi(q.z); x[6] = bf16lo(q.w); x[7] = bf16hi(q.w);
  } else {
    const uint4 q2 = __ldg(reinterpret_cast<const uint4*>(p) + 1);
    x[0] = __uint_as_float(q.x); x[1] = __uint_as_float(q.y);
    x[2] = __uint_as_float(q.z); x[3] = __uint_as_float(q.w);
    x[4] = __uint_as_float(q2.x); x[5] = __uint_as_float(q2.y);
    x[6] = __uint_as_float(q2.z); x[7] = __uint_as_float(q2.w);
  }
}

struct HeadStepParams {
  const void* E;
  const void* W;                   // gated: W_g [rank, H + rank]; RNN: [3][rank][2 rank + H]
  const float* Zh;                 // [n_split][R gamma][n_out] hidden-state partials
  int n_split, rows;               // rows = R gamma
  const int32_t* prev_tok;
  const unsigned long long* keys;  // [gamma][R_max] argmax keys of the draft steps
  float* state;                    // RNN: [2][R_max][rank]; position j writes buffer j % 2
  float* A;                        // [R, gamma, rank] the representation out
  int* status;
  int R_max, V, H, rank, gamma, act, bias_at_first;
};

// The previous token of request r at position j (the anchor at j = 0); an
// out-of-range token is reported and replaced by 0.
__device__ __forceinline__ int head_prev_token(const HeadStepParams& p, int j, int r) {
  int prev = j == 0 ? p.prev_tok[r] : (int)key_index(__ldcg(&p.keys[(size_t)(j - 1) * p.R_max + r]));
  if (prev < 0 || prev >= p.V) {
    if ((threadIdx.x & 31) == 0) set_status(p.status, kErrArg);
    prev = 0;
  }
  return prev;
}

__device__ __forceinline__ float sigmoid_f(float z) {
  return z >= 0.f ? 1.f / (1.f + expf(-z)) : expf(z) / (1.f + expf(z));
}

// Elements c .. c + 7 of the Markov row act(E[prev]) (c % 8 == 0).
template <typename T>
__device__ __forceinline__ void markov8(const HeadStepParams& p, int prev, int c, float (&m)[8]) {
  load8<T>(static_cast<const T*>(p.E) + (size_t)prev * p.rank + c, m);
#pragma unroll
  for (int e = 0; e < 8; ++e) m[e] = act_apply(m[e], p.act);
}

// Lane q's hidden-state partial base[q * stride] (q < n_split, q < 32),
// loaded ahead of the drafted-token work it does not depend on.
__device__ __forceinline__ float partial_lane(const float* base, size_t stride, int n_split) {
  const int lane = threadIdx.x & 31;
  return lane < n_split ? base[(size_t)lane * stride] : 0.f;
}

// z plus the partials base[q * stride], q = 0 .. n_split - 1, added in split
// order on lane 0: the first 32 from v0 (partial_lane), handed to lane 0 by
// shuffles in order, any further ones loaded 32 at a time the same way.
__device__ __forceinline__ float add_partials(float z, float v0, const float* base, size_t stride,
                                              int n_split) {
  const int lane = threadIdx.x & 31;
  for (int q0 = 0; q0 < n_split; q0 += 32) {
    const int q = q0 + lane;
    const float v = q0 == 0 ? v0 : (q < n_split ? base[(size_t)q * stride] : 0.f);
    const int nq = n_split - q0 < 32 ? n_split - q0 : 32;
    for (int i = 0; i < nq; ++i) z += __shfl_sync(0xffffffffu, v, i);
  }
  return z;
}

// Element k of a vector whose lane-th 8-element chunk (elements 8 lane ..
// 8 lane + 7) each lane holds in x (k < 256), on every lane.
__device__ __forceinline__ float chunk_elem(const float (&x)[8], int k) {
  // a predicated select per element (a plain select chain on one index is
  // turned into an indexed load from a stack copy of x)
  float v = x[0];
#pragma unroll
  for (int e = 1; e < 8; ++e)
    asm("{\n\t.reg .pred q;\n\tsetp.eq.s32 q, %2, %3;\n\tselp.f32 %0, %1, %0, q;\n\t}"
        : "+f"(v)
        : "f"(x[e]), "r"(k & 7), "r"(e));
  return __shfl_sync(0xffffffffu, v, (k >> 3) & 31);
}

// Whether position j carries no bias (position 0 without first-position
// bias): its representation is zero and the RNN state stays zero.
__device__ __forceinline__ bool head_unbiased(const HeadStepParams& p, int j) {
  return j == 0 && !p.bias_at_first;
}

// Gated head, outputs k0 .. k0 + NK - 1 of request r at position j:
// a[k] = g[k] * m[k].  Per output the arithmetic does not depend on NK: each
// lane multiplies its 8 columns in order, the lanes' sums meet in a
// butterfly, lane 0 adds the partials in split order.  rank <= 256: a lane
// holds at most one 8-column chunk.
template <typename T, int NK>
__device__ __forceinline__ void gate_outputs_warp(const HeadStepParams& p, int j, int r, int k0) {
  const int lane = threadIdx.x & 31;
  const size_t row = (size_t)r * p.gamma + j;
  if (head_unbiased(p, j)) {
    if (lane < NK) p.A[row * p.rank + k0 + lane] = 0.f;
    return;
  }
  float zp[NK];
#pragma unroll
  for (int i = 0; i < NK; ++i)
    zp[i] = partial_lane(p.Zh + row * p.rank + k0 + i, (size_t)p.rows * p.rank, p.n_split);
  const bool has = lane * 8 < p.rank;
  float w[NK][8];
#pragma unroll
  for (int i = 0; i < NK; ++i)
    if (has) load8<T>(static_cast<const T*>(p.W) + (size_t)(k0 + i) * (p.H + p.rank) + p.H + lane * 8, w[i]);
  const int prev = head_prev_token(p, j, r);
  float m[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (has) markov8<T>(p, prev, lane * 8, m);
#pragma unroll
  for (int i = 0; i < NK; ++i) {
    float dot = 0.f;
    if (has) {
#pragma unroll
      for (int e = 0; e < 8; ++e) dot = fmaf(w[i][e], m[e], dot);
    }
    dot = warp_sum(dot);
    const float z = add_partials(dot, zp[i], p.Zh + row * p.rank + k0 + i, (size_t)p.rows * p.rank,
                                 p.n_split);
    const float mk = chunk_elem(m, k0 + i);
    if (lane == 0) {
      if (!isfinite(z)) set_status(p.status, kErrNonfinite);
      p.A[row * p.rank + k0 + i] = sigmoid_f(z) * mk;
    }
  }
}

__device__ __forceinline__ bool rnn_first(const HeadStepParams& p, int j) {
  return j == 0 || (j == 1 && !p.bias_at_first);
}
__device__ __forceinline__ float* rnn_state_buf(const HeadStepParams& p, int j) {
  return p.state + (size_t)(j & 1) * p.R_max * p.rank;
}

// The lane's chunks of [s; m] (2 rank <= 512 columns: chunk i covers
// columns 8 lane + 256 i .. + 7): s from the state buffer (zero when s is
// null), m the Markov row.  rank % 8 == 0: no chunk straddles the halves.
template <typename T>
__device__ __forceinline__ void rnn_concat(const HeadStepParams& p, const float* s, int prev,
                                           float (&x)[2][8]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int c = lane * 8 + 256 * i;
#pragma unroll
    for (int e = 0; e < 8; ++e) x[i][e] = 0.f;
    if (c >= 2 * p.rank) continue;
    if (c >= p.rank) {
      markov8<T>(p, prev, c - p.rank, x[i]);
    } else if (s) {
      const float4 a = __ldcg(reinterpret_cast<const float4*>(s + c));
      const float4 b = __ldcg(reinterpret_cast<const float4*>(s + c) + 1);
      x[i][0] = a.x; x[i][1] = a.y; x[i][2] = a.z; x[i][3] = a.w;
      x[i][4] = b.x; x[i][5] = b.y; x[i][6] = b.z; x[i][7] = b.w;
    }
  }
}

// Dot of a weight row's first 2 rank columns with the lane chunks x, one
// warp: each lane multiplies its columns in increasing order, then a
// butterfly sum.
template <typename T>
__device__ __forceinline__ float rnn_dot(const HeadStepParams& p, const T* wrow,
                                         const float (&x)[2][8]) {
  const int lane = threadIdx.x & 31;
  float dot = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int c = lane * 8 + 256 * i;
    if (c < 2 * p.rank) {
      float w[8];
      load8<T>(wrow + c, w);
#pragma unroll
      for (int e = 0; e < 8; ++e) dot = fmaf(w[e], x[i][e], dot);
    }
  }
  return warp_sum(dot);
}

// RNN head, state units k0 .. k0 + NK - 1 of request r at position j: gate,
// candidate and the new state s_j[k].
template <typename T, int NK>
__device__ __forceinline__ void rnn_state_warp(const HeadStepParams& p, int j, int r, int k0) {
  if (head_unbiased(p, j)) return;   // no bias, the state stays zero
  const int lane = threadIdx.x & 31;
  const size_t row = (size_t)r * p.gamma + j;
  const float* zrow = p.Zh + row * 3 * p.rank;
  const size_t zs = (size_t)p.rows * 3 * p.rank;
  float zpg[NK], zpc[NK];
#pragma unroll
  for (int i = 0; i < NK; ++i) {
    zpg[i] = partial_lane(zrow + k0 + i, zs, p.n_split);
    zpc[i] = partial_lane(zrow + p.rank + k0 + i, zs, p.n_split);
  }
  const int prev = head_prev_token(p, j, r);
  const float* sp = rnn_first(p, j) ? nullptr : rnn_state_buf(p, j + 1) + (size_t)r * p.rank;
  float x[2][8];
  rnn_concat<T>(p, sp, prev, x);
  const T* Wr = static_cast<const T*>(p.W);
  const int ld = 2 * p.rank + p.H;
#pragma unroll
  for (int i = 0; i < NK; ++i) {
    const int k = k0 + i;
    const float dg = rnn_dot<T>(p, Wr + (size_t)k * ld, x);
    const float dc = rnn_dot<T>(p, Wr + (size_t)(p.rank + k) * ld, x);
    const float zg = add_partials(dg, zpg[i], zrow + k, zs, p.n_split);
    const float zc = add_partials(dc, zpc[i], zrow + p.rank + k, zs, p.n_split);
    const float s_old = chunk_elem(x[0], k);   // s[k] (k < rank <= 256), 0 at the first position
    if (lane == 0) {
      if (!isfinite(zg) || !isfinite(zc)) set_status(p.status, kErrNonfinite);
      const float g = sigmoid_f(zg);
      const float c = tanhf(zc);
      rnn_state_buf(p, j)[(size_t)r * p.rank + k] = g * s_old + (1.f - g) * c;
    }
  }
}

// RNN head, outputs k0 .. k0 + NK - 1 of request r at position j:
// o_j = tanh(W_o [s_j; m; h_j]).
template <typename T, int NK>
__device__ __forceinline__ void rnn_out_warp(const HeadStepParams& p, int j, int r, int k0) {
  const int lane = threadIdx.x & 31;
  const size_t row = (size_t)r * p.gamma + j;
  if (head_unbiased(p, j)) {
    if (lane < NK) p.A[row * p.rank + k0 + lane] = 0.f;
    return;
  }
  const float* zrow = p.Zh + row * 3 * p.rank + 2 * p.rank;
  const size_t zs = (size_t)p.rows * 3 * p.rank;
  float zp[NK];
#pragma unroll
  for (int i = 0; i < NK; ++i) zp[i] = partial_lane(zrow + k0 + i, zs, p.n_split);
  const int prev = head_prev_token(p, j, r);
  float x[2][8];
  rnn_concat<T>(p, rnn_state_buf(p, j) + (size_t)r * p.rank, prev, x);
  const T* Wr = static_cast<const T*>(p.W);
  const int ld = 2 * p.rank + p.H;
#pragma unroll
  for (int i = 0; i < NK; ++i) {
    const float d = rnn_dot<T>(p, Wr + (size_t)(2 * p.rank + k0 + i) * ld, x);
    const float z = add_partials(d, zp[i], zrow + k0 + i, zs, p.n_split);
    if (lane == 0) {
      if (!isfinite(z)) set_status(p.status, kErrNonfinite);
      p.A[row * p.rank + k0 + i] = tanhf(z);
    }
  }
}

}  // namespace dsd
