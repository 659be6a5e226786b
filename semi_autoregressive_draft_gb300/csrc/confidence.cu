// Confidence side of the scheduler's input: the confidence head, the static
// threshold truncation it replaces, and calibration metrics of the survival
// probabilities.
//
// Pages: "Qwen3.8-Flash-Next DSpark 训练实验", Confidence head 与训练目标
// (s = w_c . [h; m] + b_c with m = W_1[t_prev], c = sigmoid(s));
// "DeepSpec 训练全流程详解（以 Qwen3 + DSpark 为例）", 4.3 Propose
// (proposal_len = min(block, first position below the threshold));
// "DSpark 论文精读", 3.1 (prefix survival a = prod c, why the
// cumulative-product bias is monitored) and 5 (reliability diagram, ECE).
//
// confidence_head_kernel: one CTA per request, wpp = 2 warps per position:
//   the previous token first, then the 16-byte
//   loads of the row's hidden state (H values split over the position's
//   warps) and of the Markov row of the token (rank values, the last warp's
//   lanes) in flight together, fp32 products with w_c; then thread 0 forms
//   c = sigmoid(s) and the survival prefix products in fp64.
// threshold_keep_kernel: one thread per request.
// calibration_kernel: a grid-stride pass, one thread per request: survival
//   in fp64, reliability bin floor(a n_bins) taken in fp64 (the oracle's
//   precision), per-CTA shared-memory sums, then global fp64 sums; the last
//   CTA to finish (a ticket) forms the means, the ECE and the errors and
//   clears the sums for the next call.
#include "dsd_common.cuh"

namespace dsd {

namespace {

// 16 bytes of dtype T as fp32 values (8 for bf16, 4 for f32)
template <typename T>
__device__ __forceinline__ int chunk_to_f32(uint4 q, float* x) {
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

__device__ __forceinline__ float sigmoid_f(float z) {
  if (z >= 0.f) return 1.f / (1.f + expf(-z));
  const float e = expf(z);
  return e / (1.f + e);
}

constexpr int kHeadMaxWarps = 32;   // warps per CTA (1024 threads)
constexpr int kHeadDepth = 4;       // 16-byte loads of each operand in flight per lane

// Sum over one warp of a[v] b[v] for v in this lane's 16-byte chunks
// (first * 32 + lane) * epc + k * step, k = 0, 1, ...: the loads of up to
// kHeadDepth chunks are issued before any product.
template <typename T>
__device__ __forceinline__ float lane_dot(const T* a, const T* b, int n, int v_first, int step) {
  constexpr int epc = 16 / (int)sizeof(T);
  float acc = 0.f;
  for (int v0 = v_first; v0 < n; v0 += kHeadDepth * step) {
    uint4 qa[kHeadDepth], qb[kHeadDepth];
#pragma unroll
    for (int d = 0; d < kHeadDepth; ++d) {
      const int v = v0 + d * step;
      if (v < n) {
        qa[d] = ld_stream16(a + v);
        qb[d] = __ldg(reinterpret_cast<const uint4*>(b + v));
      }
    }
#pragma unroll
    for (int d = 0; d < kHeadDepth; ++d) {
      if (v0 + d * step < n) {
        float x[8], y[8];
        const int k = chunk_to_f32<T>(qa[d], x);
        chunk_to_f32<T>(qb[d], y);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (e < k) acc = fmaf(x[e], y[e], acc);
      }
    }
  }
  return acc;
}

template <typename T>
__global__ void __launch_bounds__(32 * kHeadMaxWarps) confidence_head_kernel(
    const T* __restrict__ h, const T* __restrict__ E, const T* __restrict__ w_c, float b_c,
    const int32_t* __restrict__ prev_tok, const int32_t* __restrict__ tokens, int H, int rank,
    int V, int gamma, int wpp, float* conf, float* survival, int* status) {
  constexpr int epc = 16 / (int)sizeof(T);
  __shared__ float s_part[kMaxGamma][kHeadMaxWarps / 2];
  const int r = blockIdx.x, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = w / wpp, part = w - j * wpp;
  if (j < gamma) {
    // the Markov row's token, loaded before anything that waits on memory
    const bool markov = part == wpp - 1;
    int t = 0;
    if (markov) {
      t = j == 0 ? prev_tok[r] : tokens[(size_t)r * gamma + j - 1];
      if (t < 0 || t >= V) {
        if (lane == 0) set_status(status, kErrArg);
        t = 0;
      }
    }
    // the Markov row's loads (rank <= 256: at most two 16-byte chunks per
    // lane) go out with the hidden state's first loads
    uint4 qe[2], qw[2];
#pragma unroll
    for (int d = 0; d < 2; ++d) {
      const int c = (lane + 32 * d) * epc;
      if (markov && c < rank) {
        qe[d] = __ldg(reinterpret_cast<const uint4*>(E + (size_t)t * rank + c));
        qw[d] = __ldg(reinterpret_cast<const uint4*>(w_c + H + c));
      }
    }
    const int step = wpp * 32 * epc;
    float v = lane_dot<T>(h + ((size_t)r * gamma + j) * H, w_c, H, (part * 32 + lane) * epc, step);
    if (markov) {
      float acc = 0.f;
#pragma unroll
      for (int d = 0; d < 2; ++d) {
        if ((lane + 32 * d) * epc < rank) {
          float x[8], y[8];
          const int k = chunk_to_f32<T>(qe[d], x);
          chunk_to_f32<T>(qw[d], y);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (e < k) acc = fmaf(x[e], y[e], acc);
        }
      }
      v += acc;
    }
    v = warp_sum(v);
    if (lane == 0) s_part[j][part] = v;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double acc = 1.0;
    for (int i = 0; i < gamma; ++i) {
      float sl = b_c;
      for (int k = 0; k < wpp; ++k) sl += s_part[i][k];
      float c = sigmoid_f(sl);
      if (!isfinite(c)) {
        set_status(status, kErrNonfinite);
        c = 0.f;
      }
      conf[(size_t)r * gamma + i] = c;
      acc *= (double)fminf(fmaxf(c, 0.f), 1.f);
      survival[(size_t)r * gamma + i] = (float)acc;
    }
  }
}

__global__ void threshold_keep_kernel(const float* conf, int R, int gamma, float threshold,
                                      int32_t* keep_len) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= R) return;
  int k = 0;
  while (k < gamma && conf[(size_t)r * gamma + k] >= threshold) ++k;   // NaN stops
  keep_len[r] = k;
}


constexpr int kCalThreads = 256;

struct CalParams {
  const float* conf;          // [M, gamma]
  const int32_t* accept_len;  // [M]
  int M, gamma, n_bins;
  double* acc;                // [2 kMaxCalBins + 2 + 2 kMaxGamma] zero between calls
  unsigned long long* cnt;    // [kMaxCalBins + 1] zero between calls (last: tested positions)
  unsigned int* ticket;       // zero between calls
  float* bins;                // [3][n_bins]: count, mean survival, mean realised survival
  float* pos;                 // [2][gamma]: mean survival, realised survival rate per position
  float* metrics;             // [4]: ece, abs_error, cumprod_bias, tested positions
  int* status;
};

// Values in [0, 1] are summed per CTA as integers in units of 2^-40 (exact
// integer atomics in shared memory; the launch gives a CTA at most 2^22
// values, below the 2^24 that would overflow 64 bits), then added to the
// fp64 sums of the grid.  The rounding, 2^-41 per value, is far below fp32.
constexpr double kFix = 1099511627776.0;   // 2^40

__device__ __forceinline__ unsigned long long to_fix(double v) { return __double2ull_rn(v * kFix); }

__global__ void __launch_bounds__(kCalThreads) calibration_kernel(CalParams p) {
  __shared__ unsigned long long sc[kMaxCalBins], sp[kMaxCalBins], spp[kMaxGamma], se;
  __shared__ unsigned int sr[kMaxCalBins], spr[kMaxGamma], st;
  __shared__ int am_last;
  const int tid = threadIdx.x;
  for (int i = tid; i < kMaxCalBins; i += kCalThreads) {
    sc[i] = sp[i] = 0ull;
    sr[i] = 0u;
  }
  if (tid < kMaxGamma) {
    spp[tid] = 0ull;
    spr[tid] = 0u;
  }
  if (tid == 0) {
    se = 0ull;
    st = 0u;
  }
  __syncthreads();
  unsigned long long err = 0ull, lp[kMaxGamma];
  unsigned int tested = 0u, lr[kMaxGamma];
  for (int j = 0; j < kMaxGamma; ++j) {
    lp[j] = 0ull;
    lr[j] = 0u;
  }
  // Every lane of a warp runs the same iterations (lanes past M take part
  // with bin -1), so the bin updates can be combined per warp: lanes with
  // the same bin add their counts and sums and one of them does the atomics.
  const int lane = tid & 31;
  for (int r0 = blockIdx.x * kCalThreads; r0 < p.M; r0 += gridDim.x * kCalThreads) {
    const int r = r0 + tid;
    const bool live = r < p.M;
    int L = live ? p.accept_len[r] : 0;
    if (L < 0 || L > p.gamma) {
      set_status(p.status, kErrArg);
      L = L < 0 ? 0 : p.gamma;
    }
    double a = 1.0;
    for (int j = 0; j < p.gamma; ++j) {
      float cf = live ? p.conf[(size_t)r * p.gamma + j] : 0.f;
      if (!isfinite(cf)) {
        set_status(p.status, kErrNonfinite);
        cf = 0.f;
      }
      const double c = (double)fminf(fmaxf(cf, 0.f), 1.f);
      a *= c;
      const unsigned int y = (live && j < L) ? 1u : 0u;
      const unsigned long long qa = live ? to_fix(a) : 0ull;
      if (live) {
        if (j <= L) {
          err += to_fix(fabs(c - (double)y));
          ++tested;
        }
        lp[j] += qa;
        lr[j] += y;
      }
      int b = (int)floor(a * (double)p.n_bins);
      b = !live ? -1 : (b < p.n_bins - 1 ? b : p.n_bins - 1);
      const unsigned peers = __match_any_sync(0xffffffffu, b);
      const unsigned n = __popc(peers);
      const unsigned ys = __reduce_add_sync(peers, y);
      const unsigned lo = __reduce_add_sync(peers, (unsigned)(qa & 0xFFFFFull));
      const unsigned hi = __reduce_add_sync(peers, (unsigned)(qa >> 20));
      if (b >= 0 && lane == __ffs(peers) - 1) {
        atomicAdd(&sc[b], (unsigned long long)n);
        atomicAdd(&sp[b], ((unsigned long long)hi << 20) + lo);
        if (ys) atomicAdd(&sr[b], ys);
      }
    }
  }
  for (int j = 0; j < p.gamma; ++j) {
    if (lp[j]) atomicAdd(&spp[j], lp[j]);
    if (lr[j]) atomicAdd(&spr[j], lr[j]);
  }
  if (err) atomicAdd(&se, err);
  if (tested) atomicAdd(&st, tested);
  __syncthreads();
  // this CTA's sums into the grid's
  for (int i = tid; i < p.n_bins; i += kCalThreads) {
    if (sc[i]) {
      atomicAdd(&p.cnt[i], sc[i]);
      atomicAdd(&p.acc[i], (double)sp[i] / kFix);
      atomicAdd(&p.acc[kMaxCalBins + i], (double)sr[i]);
    }
  }
  if (tid < p.gamma) {
    atomicAdd(&p.acc[2 * kMaxCalBins + 2 + tid], (double)spp[tid] / kFix);
    atomicAdd(&p.acc[2 * kMaxCalBins + 2 + kMaxGamma + tid], (double)spr[tid]);
  }
  if (tid == 0) {
    atomicAdd(&p.acc[2 * kMaxCalBins], (double)se / kFix);
    atomicAdd(&p.cnt[kMaxCalBins], (unsigned long long)st);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) am_last = (atomicAdd(p.ticket, 1u) == gridDim.x - 1) ? 1 : 0;
  __syncthreads();
  if (!am_last || tid != 0) return;
  __threadfence();
  const double total = (double)p.M * p.gamma;
  double ece = 0.0;
  for (int b = 0; b < p.n_bins; ++b) {
    const unsigned long long n = __ldcg(&p.cnt[b]);
    const double mp = n ? __ldcg(&p.acc[b]) / (double)n : 0.0;
    const double mr = n ? __ldcg(&p.acc[kMaxCalBins + b]) / (double)n : 0.0;
    p.bins[b] = (float)n;
    p.bins[p.n_bins + b] = (float)mp;
    p.bins[2 * p.n_bins + b] = (float)mr;
    ece += (double)n / total * fabs(mp - mr);
    p.cnt[b] = 0ull;
    p.acc[b] = 0.0;
    p.acc[kMaxCalBins + b] = 0.0;
  }
  double bias_sum = 0.0;   // sum of (a - y) over all positions
  for (int j = 0; j < p.gamma; ++j) {
    double* a = p.acc + 2 * kMaxCalBins + 2;
    bias_sum += __ldcg(&a[j]) - __ldcg(&a[kMaxGamma + j]);
    p.pos[j] = p.M ? (float)(__ldcg(&a[j]) / p.M) : 0.f;
    p.pos[p.gamma + j] = p.M ? (float)(__ldcg(&a[kMaxGamma + j]) / p.M) : 0.f;
    a[j] = a[kMaxGamma + j] = 0.0;
  }
  const unsigned long long nt = __ldcg(&p.cnt[kMaxCalBins]);
  p.metrics[0] = p.M ? (float)ece : 0.f;
  p.metrics[1] = nt ? (float)(__ldcg(&p.acc[2 * kMaxCalBins]) / (double)nt) : 0.f;
  p.metrics[2] = p.M ? (float)(bias_sum / total) : 0.f;
  p.metrics[3] = (float)nt;
  p.acc[2 * kMaxCalBins] = p.acc[2 * kMaxCalBins + 1] = 0.0;
  p.cnt[kMaxCalBins] = 0ull;
  *p.ticket = 0u;   // ready for the next call (kernels on the stream run in order)
}
}  // namespace

cudaError_t launch_confidence_head(const Ctx& ctx, const ConfHeadArgs& a, cudaStream_t s) {
  if (a.R == 0) return cudaSuccess;
  // two warps per position: two CTAs of 448 threads share an SM at gamma = 7,
  // so 256 requests run in one wave (four warps per position took two)
  const int wpp = 2;
  const dim3 grid(a.R), block(32 * wpp * a.gamma);
  if (a.dtype == 1)
    confidence_head_kernel<__nv_bfloat16><<<grid, block, 0, s>>>(
        static_cast<const __nv_bfloat16*>(a.h), static_cast<const __nv_bfloat16*>(a.E),
        static_cast<const __nv_bfloat16*>(a.w_c), a.b_c, a.prev_tok, a.tokens, a.H, a.rank, a.V,
        a.gamma, wpp, a.conf, a.survival, ctx.ws.status);
  else
    confidence_head_kernel<float><<<grid, block, 0, s>>>(
        static_cast<const float*>(a.h), static_cast<const float*>(a.E),
        static_cast<const float*>(a.w_c), a.b_c, a.prev_tok, a.tokens, a.H, a.rank, a.V, a.gamma,
        wpp, a.conf, a.survival, ctx.ws.status);
  count_launch(ctx);
  return cudaGetLastError();
}

cudaError_t launch_threshold_keep(const Ctx& ctx, int R, const float* conf, float threshold,
                                  int32_t* keep_len, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  threshold_keep_kernel<<<(R + 255) / 256, 256, 0, s>>>(conf, R, ctx.cfg.gamma, threshold, keep_len);
  count_launch(ctx);
  return cudaGetLastError();
}

cudaError_t launch_calibration(const Ctx& ctx, const CalArgs& a, cudaStream_t s) {
  CalParams p{};
  p.conf = a.conf;
  p.accept_len = a.accept_len;
  p.M = a.M;
  p.gamma = a.gamma;
  p.n_bins = a.n_bins;
  p.acc = ctx.ws.cal_acc;
  p.cnt = ctx.ws.cal_cnt;
  p.ticket = ctx.ws.tickets + 2;
  p.bins = a.bins;
  p.pos = a.pos;
  p.metrics = a.metrics;
  p.status = ctx.ws.status;
  int grid = (a.M + kCalThreads - 1) / kCalThreads;
  grid = grid < 1 ? 1 : (grid > 2 * ctx.num_sms ? 2 * ctx.num_sms : grid);
  // at most 2^22 values per CTA, so its 2^-40 fixed-point sums cannot overflow
  const long long min_grid = ((long long)a.M * a.gamma + (1 << 22) - 1) >> 22;
  if (grid < min_grid) grid = (int)min_grid;
  calibration_kernel<<<grid, kCalThreads, 0, s>>>(p);
  count_launch(ctx);
  return cudaGetLastError();
}


// ---------------------------------------------------------------------------
// AUROC of predicted survival against realised survival ("DSpark 论文精读"
// 5: the raw head's ranking quality beside its reliability diagram).  Over
// all (r, j) positions the score is a[r, j] = prod_{i <= j} clamp(conf[r, i])
// (fp64, the same sequential product as dsd_calibration) and the label
// y = (j < accept_len[r]).  AUROC = (#pairs positive > negative + 1/2 #ties)
// / (P N), 0.5 when a class is empty.
//
// Sorting instead of binning keeps it exact: each position becomes the key
// bits(a) << 1 | label bit (a >= 0, so its bits order like its value), the
// caller's scratch holds the keys padded to a power of two with all-ones
// keys, and a bitonic network sorts them in place.  With the label bit 0 for
// positives, a positive is preceded within its run of equal scores only by
// positives, so the negatives before it are those with a smaller score
// (U_low); with the bit reversed, those with a smaller or equal score
// (U_high).  U_low + U_high = 2 (#greater + 1/2 #ties) over all pairs.  The
// counts are exact integers; the division is fp64.
// ---------------------------------------------------------------------------
namespace {

constexpr int kAucTile = 1024;       // keys per shared-memory bitonic tile
constexpr int kAucThreads = 512;     // threads of the tile kernels (two keys each)

struct AucScratch {
  unsigned long long* keys;    // [n_pad]
  unsigned int* bneg;          // [n_pad / kAucTile] negatives per tile, then their exclusive scan
  unsigned long long* acc;     // [4]: U (this ordering), P, N, U_low
};

__global__ void auc_keys_kernel(const float* conf, const int32_t* accept_len, int M, int gamma,
                                int n_pad, int pos_bit, unsigned long long* keys,
                                unsigned long long* acc, int* status) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_pad; i += gridDim.x * blockDim.x) {
    if (i >= M * gamma) {
      keys[i] = ~0ull;
      continue;
    }
    const int r = i / gamma, j = i - r * gamma;
    int L = accept_len[r];
    if (L < 0 || L > gamma) {
      set_status(status, kErrArg);
      L = L < 0 ? 0 : gamma;
    }
    double a = 1.0;
    for (int t = 0; t <= j; ++t) {
      float cf = conf[(size_t)r * gamma + t];
      if (!isfinite(cf)) {
        set_status(status, kErrNonfinite);
        cf = 0.f;
      }
      a *= (double)fminf(fmaxf(cf, 0.f), 1.f);
    }
    const int y = j < L ? 1 : 0;
    const unsigned long long lbit = (unsigned long long)(y ? pos_bit : 1 - pos_bit);
    keys[i] = ((unsigned long long)__double_as_longlong(a) << 1) | lbit;
    if (pos_bit == 0) atomicAdd(&acc[y ? 1 : 2], 1ull);   // P, N: counted once
  }
}

// One comparator of the bitonic network at stage k, distance j: element i1
// and i1 + j, ascending where bit k of i1 is clear.
__device__ __forceinline__ void auc_cmp(unsigned long long& x, unsigned long long& y, bool asc) {
  if ((x > y) == asc) {
    const unsigned long long t = x;
    x = y;
    y = t;
  }
}

// Stage k, every distance j < kAucTile down to 1 (all of stages k <= kAucTile
// when sort_tile is set), within tiles of kAucTile keys in shared memory.
__global__ void __launch_bounds__(kAucThreads) auc_tile_kernel(unsigned long long* keys, int k,
                                                               int sort_tile) {
  __shared__ unsigned long long sk[kAucTile];
  const int base = blockIdx.x * kAucTile, t = threadIdx.x;
  sk[t] = keys[base + t];
  sk[t + kAucThreads] = keys[base + t + kAucThreads];
  __syncthreads();
  const int k_first = sort_tile ? 2 : k, k_last = sort_tile ? kAucTile : k;
  for (int kk = k_first; kk <= k_last; kk <<= 1) {
    for (int j = (kk >> 1) < (kAucTile >> 1) ? (kk >> 1) : (kAucTile >> 1); j >= 1; j >>= 1) {
      const int i1 = 2 * j * (t / j) + (t % j);
      auc_cmp(sk[i1], sk[i1 + j], ((base + i1) & kk) == 0);
      __syncthreads();
    }
  }
  keys[base + t] = sk[t];
  keys[base + t + kAucThreads] = sk[t + kAucThreads];
}

// Stage k, one distance j >= kAucTile over the whole array.
__global__ void auc_global_kernel(unsigned long long* keys, int n_pad, int k, int j) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < n_pad / 2; t += gridDim.x * blockDim.x) {
    const int i1 = 2 * j * (t / j) + (t % j);
    unsigned long long x = keys[i1], y = keys[i1 + j];
    auc_cmp(x, y, (i1 & k) == 0);
    keys[i1] = x;
    keys[i1 + j] = y;
  }
}

__device__ __forceinline__ bool auc_is_neg(unsigned long long key, int pos_bit) {
  return key != ~0ull && (int)(key & 1ull) != pos_bit;
}

// Negatives per tile of the sorted keys.
__global__ void __launch_bounds__(kAucThreads) auc_count_kernel(const unsigned long long* keys,
                                                                int pos_bit, unsigned int* bneg) {
  const int base = blockIdx.x * kAucTile, t = threadIdx.x;
  const int n = (auc_is_neg(keys[base + t], pos_bit) ? 1 : 0) +
                (auc_is_neg(keys[base + t + kAucThreads], pos_bit) ? 1 : 0);
  const int tot = __syncthreads_count(n & 1) + 2 * __syncthreads_count(n >> 1);
  if (t == 0) bneg[blockIdx.x] = (unsigned int)tot;
}

// Exclusive scan of the tiles' negative counts (one CTA).
__global__ void __launch_bounds__(1024) auc_scan_kernel(unsigned int* bneg, int n_tiles) {
  __shared__ unsigned long long part[1024];
  const int t = threadIdx.x;
  const int per = (n_tiles + 1023) / 1024;
  unsigned long long s = 0ull;
  for (int q = 0; q < per; ++q) {
    const int i = t * per + q;
    if (i < n_tiles) s += bneg[i];
  }
  part[t] = s;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const unsigned long long v = t >= o ? part[t - o] : 0ull;
    __syncthreads();
    part[t] += v;
    __syncthreads();
  }
  unsigned long long off = t > 0 ? part[t - 1] : 0ull;
  for (int q = 0; q < per; ++q) {
    const int i = t * per + q;
    if (i < n_tiles) {
      const unsigned int c = bneg[i];
      bneg[i] = (unsigned int)off;
      off += c;
    }
  }
}

// Sum over positives of the negatives before them in the sorted order.
__global__ void __launch_bounds__(kAucThreads) auc_sum_kernel(const unsigned long long* keys,
                                                              int pos_bit,
                                                              const unsigned int* bneg_off,
                                                              unsigned long long* acc) {
  __shared__ unsigned int wsum[kAucThreads / 32];
  const int base = blockIdx.x * kAucTile, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  // thread t holds keys base + 2t and base + 2t + 1 (consecutive)
  const unsigned long long k0 = keys[base + 2 * t], k1 = keys[base + 2 * t + 1];
  const unsigned int n0 = auc_is_neg(k0, pos_bit) ? 1u : 0u, n1 = auc_is_neg(k1, pos_bit) ? 1u : 0u;
  unsigned int incl = n0 + n1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  unsigned int woff = 0;
  for (int w = 0; w < warp; ++w) woff += wsum[w];
  const unsigned long long before = (unsigned long long)bneg_off[blockIdx.x] + woff + incl - n0 - n1;
  unsigned long long u = 0ull;
  if (k0 != ~0ull && !n0) u += before;            // a positive: the negatives before it
  if (k1 != ~0ull && !n1) u += before + n0;
  for (int o = 16; o >= 1; o >>= 1) u += __shfl_xor_sync(0xffffffffu, u, o);
  if (lane == 0 && u) atomicAdd(&acc[0], u);
}

__global__ void auc_finish_kernel(unsigned long long* acc, int phase, double* auroc) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  if (phase == 0) {            // U_low done: keep it, clear the running sum
    acc[3] = acc[0];
    acc[0] = 0ull;
    return;
  }
  const double P = (double)acc[1], N = (double)acc[2];
  *auroc = (P == 0.0 || N == 0.0) ? 0.5 : (0.5 * ((double)acc[3] + (double)acc[0])) / (P * N);
}

}  // namespace

size_t auroc_npad(int M, int gamma) {
  const long long n = (long long)M * gamma;
  long long p = kAucTile;
  while (p < n) p <<= 1;
  return (size_t)p;
}

size_t auroc_scratch_bytes(int M, int gamma) {
  const size_t n_pad = auroc_npad(M, gamma);
  return n_pad * 8 + ((n_pad / kAucTile * 4 + 255) / 256) * 256 + 64;
}

cudaError_t launch_auroc(const Ctx& ctx, int M, const float* conf, const int32_t* accept_len,
                         void* scratch, double* auroc, cudaStream_t s) {
  const int gamma = ctx.cfg.gamma;
  const int n_pad = (int)auroc_npad(M, gamma);
  const int n_tiles = n_pad / kAucTile;
  unsigned char* base = static_cast<unsigned char*>(scratch);
  AucScratch w;
  w.keys = reinterpret_cast<unsigned long long*>(base);
  w.bneg = reinterpret_cast<unsigned int*>(base + (size_t)n_pad * 8);
  w.acc = reinterpret_cast<unsigned long long*>(base + (size_t)n_pad * 8 +
                                                ((size_t)n_tiles * 4 + 255) / 256 * 256);
  cudaError_t e = cudaMemsetAsync(w.acc, 0, 4 * sizeof(unsigned long long), s);
  if (e != cudaSuccess) return e;
  const int grid_e = ctx.num_sms * 8;
  for (int pos_bit = 0; pos_bit < 2; ++pos_bit) {
    auc_keys_kernel<<<grid_e, 256, 0, s>>>(conf, accept_len, M, gamma, n_pad, pos_bit, w.keys,
                                           w.acc, ctx.ws.status);
    auc_tile_kernel<<<n_tiles, kAucThreads, 0, s>>>(w.keys, kAucTile, 1);
    count_launch(ctx, 2);
    for (int k = 2 * kAucTile; k <= n_pad; k <<= 1) {
      for (int j = k >> 1; j >= kAucTile; j >>= 1) {
        auc_global_kernel<<<grid_e, 256, 0, s>>>(w.keys, n_pad, k, j);
        count_launch(ctx);
      }
      auc_tile_kernel<<<n_tiles, kAucThreads, 0, s>>>(w.keys, k, 0);
      count_launch(ctx);
    }
    auc_count_kernel<<<n_tiles, kAucThreads, 0, s>>>(w.keys, pos_bit, w.bneg);
    auc_scan_kernel<<<1, 1024, 0, s>>>(w.bneg, n_tiles);
    auc_sum_kernel<<<n_tiles, kAucThreads, 0, s>>>(w.keys, pos_bit, w.bneg, w.acc);
    auc_finish_kernel<<<1, 32, 0, s>>>(w.acc, pos_bit, auroc);
    count_launch(ctx, 4);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dsd
