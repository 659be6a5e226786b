// tcgen05 (5th-generation tensor core) engine of dsd_propose: one launch per
// draft step for a batch of up to 256 requests, one CTA per SM.
//
// Pages: "Qwen3.8-Flash-Next DSpark 训练实验", Baseline 架构 / Markov 顺序修正
// (m_i = W_1[t_{i-1}], b_i = W_2 m_i, l_i = l_i^0 + b_i, greedy argmax over the
// full vocabulary); "DSpark notes" 2.3 (one lookup plus one low-rank
// projection per step); "DSpark 论文精读" 2.2 (x_j ~ Softmax(U_j + b)).
//
// Draft step j's bias projection for the whole batch is the GEMM
//     D[R, V] = M[R, r] * W[V, r]^T,    M[r_, :] = E[x_{r_, j-1}, :]
// with requests on the MMA's M dimension (two 128-row M-tiles for R = 256)
// and the vocabulary on N (tiles of 128).  Each CTA owns a contiguous range
// of vocabulary tiles.  Warp roles (12 warps):
//   warp 0      TMA producer of W tiles ([128 vocab x 64 K] boxes, 128-byte
//               swizzle, L2 evict-last: W stays resident across the steps)
//   warp 1      TMEM allocator and the single thread that issues tcgen05.mma
//               (M = 128, N = 128, K = 16 per instruction) into two
//               double-buffered fp32 accumulators per M-tile (512 columns)
//   warps 2, 3  TMA producers of U, one per M-tile: [128 requests x 32 vocab]
//               boxes of the [V, gamma, R] view (64-byte swizzle,
//               evict-first: U is read once), each into its own ring
//   warps 4-11  epilogue, four warps per M-tile: first they gather the A
//               operand (rows of E for the tokens chosen at step j-1) into
//               shared memory in the UMMA K-major 128-byte-swizzled layout;
//               then thread = one request row: tcgen05.ld brings 32
//               accumulator columns, U comes from shared memory, and the
//               biased logits are folded into a running base-2 log-sum-exp
//               and an argmax (greedy) or Gumbel-max (sampled) key; they never
//               leave registers.
//
// Every mbarrier has exactly one consumer role that waits on each of its
// phases in order (a parity wait cannot tell phase k from phase k + 2, so no
// waiter may skip a phase).  That is why each M-tile has its own U ring and
// producer: with one ring shared by both M-tiles, a group's consecutive waits
// on a slot would skip the other group's phase.
//
// At the end each CTA publishes per-request partials: atomicMax of the packed
// argmax key and an (m, s) log-sum-exp partial.  The next step's launch reads
// the keys, so the kernel boundary is the batch-wide synchronisation between
// steps.  Every mbarrier wait is bounded: on time-out the kernel records
// DSD_ERR_TIMEOUT, stops issuing work, waits (bounded) for its own copies in
// flight, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdio.h>

#include "dsd_common.cuh"
#include "tc_ptx.cuh"

namespace dsd {

namespace {

constexpr int kTcThreads = 384;
constexpr int kTileN = 128;          // vocabulary rows per tile (UMMA N)
constexpr int kTileM = 128;          // requests per M-tile (UMMA M)
constexpr int kMaxMT = 2;            // M-tiles per launch (R <= 256)
constexpr int kKChunk = 64;          // K elements per 128-byte swizzle row
constexpr int kMaxKC = 4;            // rank <= 256
constexpr int kWStage = 16384;       // one [128 x 64] bf16 W box
constexpr int kNB = 3;               // W ring stages
constexpr int kUCols = 32;           // vocabulary columns per U box
constexpr int kUBox = kTileM * kUCols * 2;   // 8 KB, rows of 64 bytes
constexpr int kNU = 3;               // U ring slots per M-tile
constexpr int kUPerTile = kTileN / kUCols;   // U boxes per M-tile and tile
constexpr int kTmemCols = 512;
constexpr uint32_t kIdesc = tc::idesc_bf16_f32(kTileM, kTileN);

constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kMaxMT * kMaxKC * kWStage;   // 128 KB of A
constexpr int kOffU = kOffB + kNB * kWStage;               // + 48 KB of W
constexpr int kOffBar = kOffU + kMaxMT * kNU * kUBox;      // + 48 KB of U
// bfull, bempty, ufull[2], uempty[2], accfull[2], accempty[2], aready, mmadone
constexpr int kNumBars = 2 * kNB + 2 * kMaxMT * kNU + 4 + 2;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 64 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
static_assert(kOffB % 1024 == 0 && kOffU % 1024 == 0, "swizzled boxes need aligned bases");

#ifdef DSD_TC_CHECKS
// Self-checking build: an out-of-range index records a distinct status code
// (-100 - site) and the access is skipped instead of performed.
#define TC_CHECK(cond, site) (((cond)) ? true : (set_status(p.status, -100 - (site)), false))
#else
#define TC_CHECK(cond, site) true
#endif

constexpr uint32_t kSpinLimit = 1u << 22;        // mbarrier polls before giving up

struct TcParams {
  const __nv_bfloat16* E;
  const int32_t* prev_tok;
  const uint32_t* req_id;
  unsigned long long* keys;  // [gamma][R_max]
  float2* parts;             // [gamma][n_part][R_max]
  int* status;
  int j;                     // draft position of this launch
  int R, R_max, r_off, V, rank, gamma, bias_at_first, n_part, ntiles, MT, sampled;
  float inv_T;
  uint32_t k0, k1;
};

struct Bars {
  uint64_t* bfull;      // [kNB]
  uint64_t* bempty;     // [kNB]
  uint64_t* ufull;      // [kMaxMT][kNU]
  uint64_t* uempty;     // [kMaxMT][kNU]
  uint64_t* accfull;    // [2]
  uint64_t* accempty;   // [2]
  uint64_t* aready;
  uint64_t* mmadone;
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         int* status) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort_flag) return false;
  }
  set_status(status, kErrTimeout);
  *abort_flag = 1;
  return false;
}

// Bounded wait that ignores the abort flag: used to drain copies in flight
// before the CTA exits.
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < (1u << 20); ++i)
    if (tc::mbar_try_wait(bar, parity)) return;
}

// Warp-uniform bounded wait: lane 0 polls, the verdict is broadcast, so the
// warp stays converged for the .sync.aligned tcgen05 instructions after it.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, abort_flag, status) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}
__device__ __forceinline__ bool warp_aborted(volatile int* abort_flag) {
  int a = 0;
  if ((threadIdx.x & 31) == 0) a = *abort_flag;
  return __shfl_sync(0xffffffffu, a, 0) != 0;
}

struct RowState {
  float m2, s, best_z;
  uint32_t best_v;
};

// Process 32 consecutive columns of one request row: x = acc + u (fp32),
// masked beyond V; fold into the base-2 log-sum-exp and the argmax key.
// Pairs of columns go through the packed fp32x2 pipe.
__device__ __forceinline__ void fold32(RowState& st, const uint32_t (&acc)[32],
                                       const uint4 (&u)[4], int v0, const TcParams& p,
                                       uint32_t rid) {
  float xs[32];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t w[4] = {u[c].x, u[c].y, u[c].z, u[c].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = c * 8 + 2 * e;
      const uint64_t x2 = tc::add2(tc::pack2(__uint_as_float(acc[i]), __uint_as_float(acc[i + 1])),
                                   tc::pack2(bf16lo(w[e]), bf16hi(w[e])));
      tc::unpack2(x2, xs[i], xs[i + 1]);
    }
  }
  if (v0 + 32 > p.V) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (v0 + i >= p.V) xs[i] = -INFINITY;
  }
  if (p.sampled) {
    const uint64_t t2 = tc::pack2(p.inv_T, p.inv_T);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const uint64_t x2 = tc::mul2(tc::pack2(xs[i], xs[i + 1]), t2);
      tc::unpack2(x2, xs[i], xs[i + 1]);
    }
  }
  float cm = tc::max3(xs[0], xs[1], xs[2]);
#pragma unroll
  for (int i = 3; i < 31; i += 2) cm = tc::max3(cm, xs[i], xs[i + 1]);
  cm = fmaxf(cm, xs[31]);
  const float M = fmaxf(st.m2, cm * kLog2e);
  if (M != -INFINITY) {
    const uint64_t l2 = tc::pack2(kLog2e, kLog2e);
    const uint64_t nm = tc::pack2(-M, -M);
    uint64_t s2 = tc::pack2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      float a, b;
      tc::unpack2(tc::fma2(tc::pack2(xs[i], xs[i + 1]), l2, nm), a, b);
      s2 = tc::add2(s2, tc::pack2(tc::ex2(a), tc::ex2(b)));
    }
    float slo, shi;
    tc::unpack2(s2, slo, shi);
    st.s = st.s * tc::ex2(st.m2 - M) + (slo + shi);
    st.m2 = M;
  }
  if (!p.sampled) {
    if (cm > st.best_z) {
      int idx = 31;
#pragma unroll
      for (int i = 31; i >= 0; --i)
        if (xs[i] == cm) idx = i;
      st.best_z = cm;
      st.best_v = (uint32_t)(v0 + idx);
    }
  } else {
    float zb = st.best_z;
    uint32_t vb = st.best_v;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const uint32_t v = (uint32_t)(v0 + 4 * g);
      const Philox4 ph = philox4x32_10(v >> 2, (uint32_t)p.j, rid, 0u, p.k0, p.k1);
      const float z0 = xs[4 * g + 0] + gumbel_from_word(ph.x);
      const float z1 = xs[4 * g + 1] + gumbel_from_word(ph.y);
      const float z2 = xs[4 * g + 2] + gumbel_from_word(ph.z);
      const float z3 = xs[4 * g + 3] + gumbel_from_word(ph.w);
      if (z0 > zb) { zb = z0; vb = v + 0; }
      if (z1 > zb) { zb = z1; vb = v + 1; }
      if (z2 > zb) { zb = z2; vb = v + 2; }
      if (z3 > zb) { zb = z3; vb = v + 3; }
    }
    st.best_z = zb;
    st.best_v = vb;
  }
}

__global__ void __launch_bounds__(kTcThreads, 1)
    propose_tc_kernel(const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmU, const TcParams p) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  unsigned char* sA = smem + kOffA;
  unsigned char* sB = smem + kOffB;
  unsigned char* sU = smem + kOffU;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  Bars b;
  b.bfull = bars;
  b.bempty = b.bfull + kNB;
  b.ufull = b.bempty + kNB;
  b.uempty = b.ufull + kMaxMT * kNU;
  b.accfull = b.uempty + kMaxMT * kNU;
  b.accempty = b.accfull + 2;
  b.aready = b.accempty + 2;
  b.mmadone = b.aready + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kNumBars) + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int MT = p.MT;
  const int KC = p.rank / kKChunk;
  const int j = p.j;
  const int t0 = (int)(((long long)blockIdx.x * p.ntiles) / gridDim.x);
  const int t1 = (int)(((long long)(blockIdx.x + 1) * p.ntiles) / gridDim.x);
  const int nt = t1 - t0;

  if (tid == 0) {
    for (int i = 0; i < kNB; ++i) {
      tc::mbar_init(&b.bfull[i], 1);
      tc::mbar_init(&b.bempty[i], 1);
    }
    for (int i = 0; i < kMaxMT * kNU; ++i) {
      tc::mbar_init(&b.ufull[i], 1);
      tc::mbar_init(&b.uempty[i], 4);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&b.accfull[i], 1);
      tc::mbar_init(&b.accempty[i], 4 * MT);
    }
    tc::mbar_init(b.aready, 8);
    tc::mbar_init(b.mmadone, 1);
    *abort_flag = 0;
    tc::mbar_fence_init();
    tc::fence_proxy_async_smem();
    tc::prefetch_tensormap(&tmW);
    tc::prefetch_tensormap(&tmU);
  }
  if (warp == 1) {
    __syncwarp();
    tc::tmem_alloc(tmem_holder, kTmemCols);
    tc::tmem_relinquish();
    tc::tc_fence_before();
  }
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------ W producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();
      uint32_t it = 0;
      for (int t = t0; t < t1 && !*abort_flag; ++t)
        for (int kc = 0; kc < KC; ++kc, ++it) {
          const int s = it % kNB;
          if (!wait_bar(&b.bempty[s], ((it / kNB) & 1) ^ 1, abort_flag, p.status)) break;
          tc::mbar_arrive_expect_tx(&b.bfull[s], kWStage);
          tc::tma_load_2d(sB + s * kWStage, &tmW, &b.bfull[s], kc * kKChunk, t * kTileN, pol);
        }
      // Tail: wait (bounded) for the copies issued last in each stage, then
      // for the consumer's release of every stage.  The releases are
      // tcgen05.commit arrivals, delivered to the mbarriers asynchronously when
      // the MMAs finish, so without this wait an arrival could reach this
      // CTA's shared memory after it exits.
      for (uint32_t k = (it > kNB ? it - kNB : 0); k < it; ++k)
        drain_bar(&b.bfull[k % kNB], (k / kNB) & 1);
      for (uint32_t k = (it > kNB ? it - kNB : 0); k < it; ++k)
        drain_bar(&b.bempty[k % kNB], (k / kNB) & 1);
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------- U producer of M-tile g
    const int g = warp - 2;
    if (lane == 0 && g < MT) {
      const uint64_t pol = policy_evict_first();
      uint64_t* full = b.ufull + g * kNU;
      uint64_t* empty = b.uempty + g * kNU;
      unsigned char* ring = sU + g * kNU * kUBox;
      uint32_t it = 0;
      for (int t = t0; t < t1 && !*abort_flag; ++t)
        for (int h = 0; h < kUPerTile; ++h) {
          const int vx = t * kTileN + h * kUCols;
          if (vx >= p.V) break;
          const int s = it % kNU;
          if (!wait_bar(&empty[s], ((it / kNU) & 1) ^ 1, abort_flag, p.status)) break;
          tc::mbar_arrive_expect_tx(&full[s], kUBox);
          tc::tma_load_3d(ring + s * kUBox, &tmU, &full[s], vx, j, p.r_off + g * kTileM, pol);
          ++it;
        }
      for (uint32_t k = (it > kNU ? it - kNU : 0); k < it; ++k)
        drain_bar(&full[k % kNU], (k / kNU) & 1);
      for (uint32_t k = (it > kNU ? it - kNU : 0); k < it; ++k)
        drain_bar(&empty[k % kNU], (k / kNU) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t bit = 0, tcount = 0;
      bool ok = wait_bar(b.aready, 0, abort_flag, p.status);
      tc::tc_fence_after();
      for (int t = t0; t < t1 && ok; ++t, ++tcount) {
        const int buf = tcount & 1;
        ok = wait_bar(&b.accempty[buf], ((tcount >> 1) & 1) ^ 1, abort_flag, p.status);
        if (!ok) break;
        tc::tc_fence_after();
        for (int kc = 0; kc < KC; ++kc, ++bit) {
          const int s = bit % kNB;
          ok = wait_bar(&b.bfull[s], (bit / kNB) & 1, abort_flag, p.status);
          if (!ok) break;
          tc::tc_fence_after();
          const uint32_t b_base = tc::smem_u32(sB + s * kWStage);
          for (int m = 0; m < MT; ++m) {
            const uint32_t d_tmem = tmem_base + (uint32_t)((buf * 2 + m) * kTileN);
            const uint32_t a_base = tc::smem_u32(sA + (m * kMaxKC + kc) * kWStage);
#pragma unroll
            for (int ks = 0; ks < kKChunk / 16; ++ks) {
              tc::umma_bf16(d_tmem, tc::sdesc_kmajor_sw128(a_base + ks * 32),
                            tc::sdesc_kmajor_sw128(b_base + ks * 32), kIdesc,
                            (kc | ks) != 0 ? 1u : 0u);
            }
          }
          tc::umma_commit(&b.bempty[s]);
        }
        if (ok) tc::umma_commit(&b.accfull[buf]);
      }
      // all issued MMAs complete before TMEM is released
      tc::umma_commit(b.mmadone);
      drain_bar(b.mmadone, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------ epilogue
    const int e = warp - 4;          // 0..7
    const int g = e >> 2;            // M-tile of this warp
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;   // row within the M-tile
    const int r = p.r_off + g * kTileM + row;
    const bool active = g < MT;
    const bool valid = active && r < p.R;
    const uint32_t rid = valid ? (p.req_id ? p.req_id[r] : (uint32_t)r) : 0u;
    const int rows_total = MT * kTileM;

    // ---- A operand: rows of E for the tokens of step j-1 ----
    // This warp fills rows e, e+8, ...: lane k fetches the token of row e+8k,
    // then rows are copied 16 at a time (16 loads in flight per lane) into
    // the 128-byte-swizzled K-major layout of the UMMA descriptors.
    {
      const bool biased = (j > 0) || p.bias_at_first;
      const int rows_per_warp = rows_total / 8;
      int my_tok = -1;
      if (lane < rows_per_warp) {
        const int rr = p.r_off + e + 8 * lane;
        if (biased && rr < p.R) {
          int tk = (j == 0) ? p.prev_tok[rr]
                            : (int)key_index(__ldcg(&p.keys[(size_t)(j - 1) * p.R_max + rr]));
          if (tk < 0 || tk >= p.V) {
            set_status(p.status, kErrArg);
            tk = 0;
          }
          my_tok = tk;
        }
      }
      const int cpr = p.rank / 8;    // 16-byte chunks per row
      for (int k0 = 0; k0 < rows_per_warp; k0 += 16) {
        uint4 v[16];
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const int tok = __shfl_sync(0xffffffffu, my_tok, (k0 + kk) & 31);
          v[kk] = make_uint4(0u, 0u, 0u, 0u);
          if (k0 + kk < rows_per_warp && tok >= 0 && lane < cpr &&
              TC_CHECK((size_t)tok * p.rank + lane * 8 + 8 <= (size_t)p.V * p.rank, 2))
            v[kk] = __ldcg(reinterpret_cast<const uint4*>(p.E + (size_t)tok * p.rank + lane * 8));
        }
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const int ri = e + 8 * (k0 + kk);
          if (k0 + kk >= rows_per_warp || lane >= cpr) continue;
          const int mt = ri / kTileM, ir = ri % kTileM;
          const int kc = lane >> 3, cc = lane & 7;
          const size_t off = (size_t)(mt * kMaxKC + kc) * kWStage + ir * 128 +
                             ((cc ^ (ir & 7)) << 4);
          if (TC_CHECK(off + 16 <= (size_t)kMaxMT * kMaxKC * kWStage, 1))
            *reinterpret_cast<uint4*>(sA + off) = v[kk];
        }
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(b.aready);
    }

    // ---- tiles ----
    RowState st{-INFINITY, 0.f, -INFINITY, 0u};
    uint64_t* full = b.ufull + g * kNU;
    uint64_t* empty = b.uempty + g * kNU;
    const unsigned char* ring = sU + g * kNU * kUBox;
    uint32_t tcount = 0, uit = 0;
    for (int tt = 0; tt < nt && active; ++tt, ++tcount) {
      if (warp_aborted(abort_flag)) break;
      const int t = t0 + tt;
      const int buf = tcount & 1;
      if (!warp_wait(&b.accfull[buf], (tcount >> 1) & 1, abort_flag, p.status)) break;
      tc::tc_fence_after();
      for (int h = 0; h < kUPerTile; ++h) {
        const int vx = t * kTileN + h * kUCols;
        if (vx >= p.V) break;
        const int s = uit % kNU;
        if (!warp_wait(&full[s], (uit / kNU) & 1, abort_flag, p.status)) break;
        // 64-byte swizzle: 16-byte chunk c of row `row` sits at chunk
        // c ^ ((row >> 1) & 3) of that row.
        const unsigned char* urow = ring + s * kUBox + row * (kUCols * 2);
        uint4 u[4];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          u[c] = *reinterpret_cast<const uint4*>(urow + ((c ^ ((row >> 1) & 3)) << 4));
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[s]);   // the slot's data is in registers
        ++uit;
        __syncwarp();
        uint32_t acc[32];
        tc::tmem_ld_32x32b_x32_wait(tmem_base + ((uint32_t)(q * 32) << 16) +
                                        (uint32_t)((buf * 2 + g) * kTileN + h * kUCols),
                                    acc);
        fold32(st, acc, u, vx, p, rid);
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&b.accempty[buf]);
    }

    // ---- publish this CTA's partials of step j ----
    if (valid && TC_CHECK(blockIdx.x < (unsigned)p.n_part && r < p.R_max, 5)) {
      atomicMax(&p.keys[(size_t)j * p.R_max + r], make_key(st.best_z, st.best_v));
      p.parts[((size_t)j * p.n_part + blockIdx.x) * p.R_max + r] = make_float2(st.m2, st.s);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

}  // namespace

int tc_supported(const Ctx& ctx, char* why, size_t why_len) {
  if (ctx.cfg.dtype != 1) {
    snprintf(why, why_len, "tcgen05 engine needs bf16 tables");
    return 0;
  }
  if (ctx.cfg.rank % kKChunk != 0 || ctx.cfg.rank > kMaxKC * kKChunk) {
    snprintf(why, why_len, "tcgen05 engine needs a Markov rank that is a multiple of 64, <= 256");
    return 0;
  }
  if (ctx.cfg.act != kActNone) {
    snprintf(why, why_len, "tcgen05 engine runs without an activation (bf16 operands)");
    return 0;
  }
  if (!encode_fn()) {
    snprintf(why, why_len, "cuTensorMapEncodeTiled is not available from the driver");
    return 0;
  }
  int smem = 0;
  cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, ctx.cfg.device);
  if (smem < kSmemBytes) {
    snprintf(why, why_len, "device lacks %d bytes of shared memory per block", kSmemBytes);
    return 0;
  }
  return 1;
}

int tc_grid(const Ctx& ctx) {
  const int ntiles = (ctx.cfg.V + kTileN - 1) / kTileN;
  return ntiles < ctx.num_sms ? ntiles : ctx.num_sms;
}

cudaError_t launch_propose_tc(const Ctx& ctx, const ProposeArgs& a, cudaStream_t s) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap tmW, tmU;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)a.rank, (cuuint64_t)a.V};
    const cuuint64_t strides[1] = {(cuuint64_t)a.rank * 2};
    const cuuint32_t box[2] = {kKChunk, kTileN};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.W), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)a.V, (cuuint64_t)a.gamma, (cuuint64_t)a.R};
    const cuuint64_t strides[2] = {(cuuint64_t)a.V * 2, (cuuint64_t)a.V * 2 * a.gamma};
    const cuuint32_t box[3] = {kUCols, 1, kTileM};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&tmU, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.U), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaMemsetAsync(ctx.ws.keys, 0,
                                  sizeof(unsigned long long) * (size_t)a.gamma * ctx.cfg.R_max, s);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(propose_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes);
  if (e != cudaSuccess) return e;

  TcParams p{};
  p.E = static_cast<const __nv_bfloat16*>(a.E);
  p.prev_tok = a.prev_tok;
  p.req_id = a.req_id;
  p.keys = ctx.ws.keys;
  p.parts = ctx.ws.lse_parts;
  p.status = ctx.ws.status;
  p.R = a.R;
  p.R_max = ctx.cfg.R_max;
  p.V = a.V;
  p.rank = a.rank;
  p.gamma = a.gamma;
  p.bias_at_first = a.bias_at_first;
  p.n_part = ctx.n_part;
  p.ntiles = (a.V + kTileN - 1) / kTileN;
  p.sampled = a.temperature > 0.f ? 1 : 0;
  p.inv_T = a.temperature > 0.f ? 1.f / a.temperature : 1.f;
  p.k0 = (uint32_t)(a.seed & 0xFFFFFFFFull);
  p.k1 = (uint32_t)(a.seed >> 32);
  const int grid = tc_grid(ctx);
  const int groups = (a.R + kMaxMT * kTileM - 1) / (kMaxMT * kTileM);

  // Steps in order; within a step, request groups of <= 256 are independent.
  for (int j = 0; j < a.gamma; ++j) {
    p.j = j;
    for (int gi = 0; gi < groups; ++gi) {
      p.r_off = gi * kMaxMT * kTileM;
      const int rem = a.R - p.r_off;
      p.MT = rem > kTileM ? 2 : 1;
      propose_tc_kernel<<<grid, kTcThreads, kSmemBytes, s>>>(tmW, tmU, p);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      count_launch(ctx);
    }
  }
  return cudaSuccess;
}

}  // namespace dsd
