// Device helpers shared by the kernels of the draft/verify hot path.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsd_internal.h"

namespace dsd {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// Element loads.  bf16 -> fp32 is exact (the bf16 bits are the high half).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ld_elem(const float* p, size_t i) { return __ldg(p + i); }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// L2 cache policies: evict-first for rows read exactly once (U, P, Q),
// evict-last for tables reused across steps and CTAs (W, E).  The policy is
// a constant, so these are plain (non-volatile) asm the compiler can hoist
// out of loops instead of re-creating it for every load.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// Streaming 16-byte load of read-only data: no L1 allocation, evict-first
// in L2.  Not volatile: the compiler may schedule independent loads early.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p), "l"(policy_evict_first()));
  return r;
}
// 16-byte load kept in L2 (reused tables: W, E).
__device__ __forceinline__ uint4 ld_keep16(const void* p) {
  uint4 r;
  asm("ld.global.nc.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p), "l"(policy_evict_last()));
  return r;
}

// ---------------------------------------------------------------------------
// Philox4x32-10 from its published definition (Salmon, Moraes, Dror, Shaw,
// SC'11): 10 rounds of two 32x32->64 multiplies with the high/low halves
// crossed over and xored with the key; the key advances by a Weyl sequence.
// ---------------------------------------------------------------------------
struct Philox4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2,
                                                  uint32_t c3, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t lo0 = 0xD2511F53u * c0;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0;
    const uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return Philox4{c0, c1, c2, c3};
}

__device__ __forceinline__ uint32_t philox_pick(const Philox4& p, int i) {
  return i == 0 ? p.x : (i == 1 ? p.y : (i == 2 ? p.z : p.w));
}

// u = ((w >> 9) + 0.5) * 2^-23: exact in fp32, strictly inside (0, 1).
// No integer-to-float conversion (a slow-pipe instruction): the 23 bits k
// become the mantissa of 1 + k 2^-23, and subtracting 1 - 2^-24 (exact in
// fp32) leaves (2k + 1) 2^-24, which has at most 24 significant bits, so
// the subtraction is exact.
__device__ __forceinline__ float uniform_from_word(uint32_t w) {
  return __uint_as_float((w >> 9) | 0x3F800000u) - 0.999999940395355224609375f;
}

// Hardware base-2 logarithm (MUFU): absolute error about 2^-22 for
// arguments in [0.5, 2], relative error about 2^-22 elsewhere.
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log2(1 - 2^d) for d < 0: the log of the residual p - q = p (1 - 2^d) with
// d = log2 q - log2 p.  For d > -1/2 (p within a factor of sqrt 2 of q),
// 1 - 2^d = -(e^u - 1) with u = d ln 2 in (-0.35, 0), from the Taylor series
// of e^u - 1 to u^7 / 5040 (the rest is below u^8 / 40320, 5e-9), which keeps
// the relative accuracy as p approaches q; below it 1 - 2^d >= 0.29 comes
// from the hardware 2^x.  Then the hardware base-2 logarithm.
__device__ __forceinline__ float log2_one_minus_exp2(float d) {
  const float u = d * 0.6931471805599453f;
  const float em1 =
      u * (1.f + u * (0.5f + u * (1.f / 6.f + u * (1.f / 24.f +
                                  u * (1.f / 120.f + u * (1.f / 720.f + u * (1.f / 5040.f)))))));
  float e2;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e2) : "f"(d));
  return lg2_approx(d > -0.5f ? -em1 : 1.f - e2);
}

// t = -ln u of a Philox word, u = ((w >> 9) + 0.5) 2^-23 (an Exp(1) draw).
// For u <= 15/16 from the hardware logarithm, whose absolute error there is
// at most 2^-22 against |log2 u| >= 0.093, so t is within a relative 3e-6;
// above 15/16 (w >= 15 2^28) from the Taylor series of -ln(1 - d) in
// d = 1 - u (exact in fp32 by Sterbenz' lemma), six terms, truncated below
// d^7/7 < 2^-26 of t.  The smallest t (the draws that win a race) come from
// the series, accurate to fp32 rounding.
__device__ __forceinline__ float neg_ln_uniform(uint32_t w) {
  constexpr float kLn2f = 0.6931471805599453f;
  const float u = uniform_from_word(w);
  if (w >= (15u << 28)) {   // u > 15/16
    const float d = 1.f - u;
    return d * (1.f + d * (0.5f + d * (1.f / 3.f + d * (0.25f + d * (0.2f + d * (1.f / 6.f))))));
  }
  return -kLn2f * lg2_approx(u);
}

// Gumbel noise g = -ln(-ln u) of a Philox word: t = -ln u as above, then
// g = -ln t from the hardware logarithm, within about 3e-6.
__device__ __forceinline__ float gumbel_from_word(uint32_t w) {
  return -0.6931471805599453f * lg2_approx(neg_ln_uniform(w));
}

// ---------------------------------------------------------------------------
// Order-preserving float <-> u32 map and the packed argmax key:
// key = ord(z) << 32 | ~index, so the unsigned maximum is the largest z and,
// among equal z, the lowest index.  A key of 0 is below every real key.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t f2ord(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float ord2f(uint32_t o) {
  const uint32_t b = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(b);
}
__device__ __forceinline__ unsigned long long make_key(float z, uint32_t idx) {
  return ((unsigned long long)f2ord(z) << 32) | (unsigned long long)(~idx);
}
__device__ __forceinline__ uint32_t key_index(unsigned long long k) {
  return ~(uint32_t)(k & 0xFFFFFFFFull);
}
__device__ __forceinline__ float key_value(unsigned long long k) { return ord2f((uint32_t)(k >> 32)); }

// ---------------------------------------------------------------------------
// Online log-sum-exp state in base 2: (m, s) stands for s * 2^m, where m is a
// maximum of log2e-scaled logits.  s = 0, m = -inf is the empty state.
// ---------------------------------------------------------------------------
struct Lse2 {
  float m, s;
};
__device__ __forceinline__ Lse2 lse2_empty() { return Lse2{-INFINITY, 0.f}; }
__device__ __forceinline__ Lse2 lse2_merge(Lse2 a, Lse2 b) {
  const float M = fmaxf(a.m, b.m);
  if (M == -INFINITY) return Lse2{M, 0.f};
  return Lse2{M, a.s * exp2f(a.m - M) + b.s * exp2f(b.m - M)};
}
// natural-log value of the state
__device__ __forceinline__ float lse2_value(Lse2 a) { return (a.m + log2f(a.s)) * kLn2; }

__device__ __forceinline__ Lse2 warp_lse2(Lse2 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Lse2 w{__shfl_xor_sync(0xffffffffu, v.m, o), __shfl_xor_sync(0xffffffffu, v.s, o)};
    v = lse2_merge(v, w);
  }
  return v;
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Record the first device-side error of a call sequence.
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float act_apply(float m, int act) {
  return act == kActSilu ? m / (1.f + __expf(-m)) : m;
}

}  // namespace dsd
