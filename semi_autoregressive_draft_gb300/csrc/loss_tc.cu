// Teacher-forced DSpark loss forward on the tcgen05 tensor cores.
//
// Pages: "DSpark 论文精读：置信度调度推测解码、半自回归生成与大模型推理加速",
// section 4.1 (position-decayed weights w_j = exp(-j / decay), the L1
// alignment term, the confidence head's BCE against the soft accept rate);
// "DeepSpec 训练全流程详解（以 Qwen3 + DSpark 为例）", section 3.4
// (compute_dspark_loss: CE, L1 = sum |p - q|, accept = 1 - L1/2, BCE with
// logits, total = 0.1 CE + 0.9 L1 + 1.0 BCE); "Qwen3.8-Flash-Next DSpark
// 训练实验", Markov 顺序修正 (l = l^0 + W_2 W_1[t_prev]).
//
// Row n = b * gamma + j of a batch of B blocks has known previous token
// prev_tok[n] (teacher forcing), so the Markov bias of every row is one GEMM
//     D[rows, V] = A[rows, r] * W[V, r]^T,   A[n, :] = E[prev_tok[n], :]
// with no sequential dependency.  The draft logits l = U + D never reach HBM.
//
// The L1 distance between two softmaxes needs both normalisers before any
// term |p_v - q_v| can be summed, so the forward takes two passes over the
// vocabulary (a streaming algorithm cannot avoid the second read: the
// biased logits of a batch are far larger than on-chip memory and L2):
//   pass 1: per (row, vocabulary range) base-2 log-sum-exp partials of l and
//           of P, and l at the target token (written by the one CTA whose
//           range holds it);
//   pass 2: each row merges its partials into log2-normalisers, then the
//           partial sums of |2^(P log2e - lp) - 2^(l log2e - lq)| per range;
//   finalize (loss_finalize_kernel): per-row L1, accept, CE and BCE, and the
//           position-weighted batch losses summed in fp64.
// Pass 2 is launched with a programmatic dependency on pass 1: its grid
// initialises, allocates TMEM, gathers A and starts streaming while pass 1
// drains, and waits for pass 1's partials only before its first tile.  It
// walks each range's tiles in reverse, so it starts on the tiles pass 1 read
// last, which may still be in L2.
//
// Grid: (M-tiles of 128 rows) x (vocabulary ranges), one CTA per SM; the
// M-tiles of one range read the same W tiles at about the same time, so all
// but the first read them from L2.  Warp roles (12 warps):
//   warp 0      TMA producer of W ([128 vocab x 64 K] boxes, 128-byte
//               swizzle), 2-stage ring of two boxes per stage (64 KB)
//   warp 1      TMEM allocator and MMA issuer: M = 128, N = 128, K = 16 per
//               tcgen05.mma with A read from TMEM, into three fp32
//               accumulators of 128 columns
//   warps 2, 3  TMA producers of U and P, one per 64-column half of a tile;
//               each ring slot holds the U box and the P box of one half
//               (2 slots per half, 128 KB)
//   warps 4-11  epilogue: first they gather A (rows of E) into TMEM columns
//               0..127 with tcgen05.st; then thread = one row and 64 columns
//               of each tile, in chunks of 32 accumulator columns.
// A in TMEM instead of shared memory is what leaves room for the P ring.
//
// Every mbarrier has exactly one consumer role that waits on each of its
// phases in order, and every wait is bounded (tc_common.cuh).
#include <math.h>
#include <stdio.h>

#include "tc_common.cuh"

namespace dsd {

namespace {

constexpr int kLThreads = 384;
constexpr int kTileN = 128;          // vocabulary columns per tile (UMMA N)
constexpr int kTileM = 128;          // rows per M-tile (UMMA M)
constexpr int kKChunk = 64;          // K elements per 128-byte swizzle row
constexpr int kMaxKC = 4;            // rank <= 256
constexpr int kBox = 16384;          // one [128 x 64] bf16 box
constexpr int kCPS = 2;              // W boxes per ring stage
constexpr int kNB = 2;               // W ring stages
constexpr int kHalf = 64;            // vocabulary columns per U / P box
constexpr int kNU = 2;               // U+P slots per column half
constexpr int kSlot = 2 * kBox;      // U box, then P box
constexpr int kNAcc = 3;             // accumulators of kTileN columns
constexpr int kAcol = 0;             // A operand: TMEM columns [0, 128)
constexpr int kDcol = 128;           // accumulators: TMEM columns [128, 512)
constexpr int kTmemCols = 512;
constexpr uint32_t kIdesc = tc::idesc_bf16_f32(kTileM, kTileN);

constexpr int kOffB = 0;
constexpr int kOffU = kOffB + kNB * kCPS * kBox;        // 64 KB of W
constexpr int kOffX = kOffU + 2 * kNU * kSlot;          // + 128 KB of U and P
constexpr int kOffBar = kOffX + kTileM * 16;            // + the halves' exchange
// bfull, bempty, ufull[2], uempty[2], accfull, accempty, aready, mmadone
constexpr int kNumBars = 2 * kNB + 4 * kNU + 2 * kNAcc + 2;
constexpr int kLossSmemBytes = kOffBar + kNumBars * 8 + 64 + 1024;  // + alignment slack
static_assert(kLossSmemBytes <= 232448, "shared memory budget of one CTA");
static_assert(kOffU % 1024 == 0 && kSlot % 1024 == 0, "swizzled boxes need aligned bases");
static_assert(kDcol + kNAcc * kTileN == kTmemCols, "TMEM: A plus the accumulators");
static_assert(kMaxKC * kKChunk / 2 <= kDcol - kAcol, "A fits its TMEM columns");

struct LossParams {
  const __nv_bfloat16* E;
  const int32_t* prev_tok;   // [rows]
  const int32_t* target;     // [rows]
  float4* parts1;            // [n_vr][rows_max] (m2 of l, s of l, m2 of P, s of P)
  float* parts2;             // [n_vr][rows_max] partial L1
  float* ltgt;               // [rows] l at the target token
  int* status;
  int rows, rows_max, V, rank, gamma, bias_at_first, n_vr, ntiles;
};

struct LossBars {
  uint64_t* bfull;      // [kNB]
  uint64_t* bempty;     // [kNB]
  uint64_t* ufull;      // [2][kNU]
  uint64_t* uempty;     // [2][kNU]
  uint64_t* accfull;    // [kNAcc]
  uint64_t* accempty;   // [kNAcc]
  uint64_t* aready;
  uint64_t* mmadone;
};

// x = u (bf16, widened exactly) + acc (fp32) for the two halves of one
// 32-bit word of U.
__device__ __forceinline__ void add_bf16x2(uint32_t w, uint32_t a_lo, uint32_t a_hi, float& lo,
                                           float& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "add.rn.f32.bf16 %0, l, %3;\n\tadd.rn.f32.bf16 %1, h, %4;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(w), "f"(__uint_as_float(a_lo)), "f"(__uint_as_float(a_hi)));
}

// Largest jump of the running base-2 maximum that is folded without
// rescaling: terms of the running sum stay below 2^kLagBits.
constexpr float kLagBits = 8.f;

// Fold 32 logits (natural scale; -inf for masked columns) into the base-2
// log-sum-exp state (m2, s), sum = s * 2^m2.  The reference m2 is raised
// only when the chunk maximum exceeds it by more than kLagBits, so the
// exponentials need not wait for the chunk maximum.  NaN or +inf inputs make
// s non-finite, which the finalize kernel reports.
__device__ __forceinline__ void lse_fold32(Lse2& st, const float (&x)[32]) {
  float gm[8];
#pragma unroll
  for (int g = 0; g < 8; ++g)
    gm[g] = fmaxf(tc::max3(x[4 * g], x[4 * g + 1], x[4 * g + 2]), x[4 * g + 3]);
  const float cm = fmaxf(tc::max3(gm[0], gm[1], gm[2]),
                         fmaxf(tc::max3(gm[3], gm[4], gm[5]), fmaxf(gm[6], gm[7])));
  const float cm2 = cm * kLog2e;
  if (cm2 > st.m + kLagBits) {
    st.s *= tc::ex2(st.m - cm2);     // 0 while the state is empty
    st.m = cm2;
  }
  if (st.m != -INFINITY) {
    const uint64_t l2 = tc::pack2(kLog2e, kLog2e);
    const uint64_t nm = tc::pack2(-st.m, -st.m);
    uint64_t e2[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float a, b;
      tc::unpack2(tc::fma2(tc::pack2(x[2 * i], x[2 * i + 1]), l2, nm), a, b);
      e2[i] = tc::pack2(tc::ex2(a), tc::ex2(b));
    }
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) e2[i] = tc::add2(e2[i], e2[i + w]);
    float slo, shi;
    tc::unpack2(e2[0], slo, shi);
    st.s += slo + shi;
  }
}

// Sum over 32 columns of |p - q| with p = 2^(xp log2e - lp2) and
// q = 2^(xq log2e - lq2) (lp2, lq2: base-2 log-normalisers).  Masked columns
// (-inf in both) contribute 0.
__device__ __forceinline__ float l1_chunk32(const float (&xq)[32], const float (&xp)[32], float lq2,
                                            float lp2) {
  const uint64_t l2 = tc::pack2(kLog2e, kLog2e);
  const uint64_t nq = tc::pack2(-lq2, -lq2);
  const uint64_t np = tc::pack2(-lp2, -lp2);
  float t[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float qa, qb, pa, pb;
    tc::unpack2(tc::fma2(tc::pack2(xq[2 * i], xq[2 * i + 1]), l2, nq), qa, qb);
    tc::unpack2(tc::fma2(tc::pack2(xp[2 * i], xp[2 * i + 1]), l2, np), pa, pb);
    t[i] = fabsf(tc::ex2(pa) - tc::ex2(qa)) + fabsf(tc::ex2(pb) - tc::ex2(qb));
  }
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] += t[i + w];
  return t[0];
}

// 128-byte swizzle: 16-byte chunk c of row `row` of a [128 x 64] bf16 box
// sits at chunk c ^ (row & 7) of that row.
__device__ __forceinline__ uint4 box_chunk(const unsigned char* box, int row, int c) {
  return *reinterpret_cast<const uint4*>(box + row * 128 + ((c ^ (row & 7)) << 4));
}

template <int kPass>
__global__ void __launch_bounds__(kLThreads, 1)
    loss_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmU,
                   const __grid_constant__ CUtensorMap tmP, const LossParams p) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  unsigned char* sB = smem + kOffB;
  unsigned char* sU = smem + kOffU;
  float4* xch = reinterpret_cast<float4*>(smem + kOffX);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  LossBars b;
  b.bfull = bars;
  b.bempty = b.bfull + kNB;
  b.ufull = b.bempty + kNB;
  b.uempty = b.ufull + 2 * kNU;
  b.accfull = b.uempty + 2 * kNU;
  b.accempty = b.accfull + kNAcc;
  b.aready = b.accempty + kNAcc;
  b.mmadone = b.aready + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kNumBars) + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int KC = p.rank / kKChunk;
  const int mt = blockIdx.x / p.n_vr;
  const int vr = blockIdx.x % p.n_vr;
  const int r0 = mt * kTileM;        // first row of this CTA's M-tile
  const int t0 = (int)(((long long)vr * p.ntiles) / p.n_vr);
  const int t1 = (int)(((long long)(vr + 1) * p.ntiles) / p.n_vr);
  const int nt = t1 - t0;
  // pass 1 walks the range forward, pass 2 backward; every role uses this map
  auto tile_of = [&](int tt) { return kPass == 1 ? t0 + tt : t1 - 1 - tt; };

  // The next grid (pass 2 after pass 1) may start on SMs as this one's CTAs
  // exit; it waits for this grid's results in griddepcontrol.wait.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int i = 0; i < kNB; ++i) {
      tc::mbar_init(&b.bfull[i], 1);
      tc::mbar_init(&b.bempty[i], 1);
    }
    for (int i = 0; i < 2 * kNU; ++i) {
      tc::mbar_init(&b.ufull[i], 1);
      tc::mbar_init(&b.uempty[i], 4);
    }
    for (int i = 0; i < kNAcc; ++i) {
      tc::mbar_init(&b.accfull[i], 1);
      tc::mbar_init(&b.accempty[i], 8);
    }
    tc::mbar_init(b.aready, 8);
    tc::mbar_init(b.mmadone, 1);
    *abort_flag = 0;
    tc::mbar_fence_init();
    tc::fence_proxy_async_smem();
    tc::prefetch_tensormap(&tmW);
    tc::prefetch_tensormap(&tmU);
    tc::prefetch_tensormap(&tmP);
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
      for (int tt = 0; tt < nt && !*abort_flag; ++tt) {
        const int t = tile_of(tt);
        for (int k0 = 0; k0 < KC; k0 += kCPS, ++it) {
          const int s = it % kNB;
          const int nch = KC - k0 < kCPS ? KC - k0 : kCPS;
          if (!wait_bar(&b.bempty[s], ((it / kNB) & 1) ^ 1, abort_flag, p.status)) break;
          tc::mbar_arrive_expect_tx(&b.bfull[s], (uint32_t)(nch * kBox));
          for (int c = 0; c < nch; ++c)
            tc::tma_load_2d(sB + (s * kCPS + c) * kBox, &tmW, &b.bfull[s], (k0 + c) * kKChunk,
                            t * kTileN, pol);
        }
      }
      // Tail: wait (bounded) for the copies issued last in each stage, then
      // for the MMAs' release of every stage (tcgen05.commit arrivals land
      // asynchronously; none may reach shared memory after the CTA exits).
      for (uint32_t k = (it > kNB ? it - kNB : 0); k < it; ++k)
        drain_bar(&b.bfull[k % kNB], (k / kNB) & 1);
      for (uint32_t k = (it > kNB ? it - kNB : 0); k < it; ++k)
        drain_bar(&b.bempty[k % kNB], (k / kNB) & 1);
    }
  } else if (warp == 2 || warp == 3) {
    // -------------------------------- U and P producer of column half hs
    const int hs = warp - 2;
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      uint64_t* full = b.ufull + hs * kNU;
      uint64_t* empty = b.uempty + hs * kNU;
      unsigned char* ring = sU + hs * kNU * kSlot;
      uint32_t it = 0;
      for (int tt = 0; tt < nt && !*abort_flag; ++tt) {
        const int vx = tile_of(tt) * kTileN + hs * kHalf;
        if (vx >= p.V) continue;           // the epilogue skips the same half
        const int s = it % kNU;
        if (!wait_bar(&empty[s], ((it / kNU) & 1) ^ 1, abort_flag, p.status)) break;
        tc::mbar_arrive_expect_tx(&full[s], kSlot);
        tc::tma_load_2d(ring + s * kSlot, &tmU, &full[s], vx, r0, pol);
        tc::tma_load_2d(ring + s * kSlot + kBox, &tmP, &full[s], vx, r0, pol);
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
      uint32_t bit = 0;
      bool ok = wait_bar(b.aready, 0, abort_flag, p.status);
      tc::tc_fence_after();   // the epilogue's TMEM stores of A are complete
      // Descriptor of the first W box; the others differ only in the
      // start-address field (16-byte units, no carry: shared memory < 2^18).
      const uint64_t db0 = tc::sdesc_kmajor_sw128(tc::smem_u32(sB));
      for (int tt = 0; tt < nt && ok; ++tt) {
        const int buf = tt % kNAcc;
        ok = wait_bar(&b.accempty[buf], ((tt / kNAcc) & 1) ^ 1, abort_flag, p.status);
        if (!ok) break;
        tc::tc_fence_after();    // the epilogue's TMEM reads of this buffer are done
        const uint32_t d_tmem = tmem_base + (uint32_t)(kDcol + buf * kTileN);
        for (int k0 = 0; k0 < KC; k0 += kCPS, ++bit) {
          const int s = bit % kNB;
          const int nch = KC - k0 < kCPS ? KC - k0 : kCPS;
          ok = wait_bar(&b.bfull[s], (bit / kNB) & 1, abort_flag, p.status);
          if (!ok) break;
          for (int c = 0; c < nch; ++c) {
            const int kc = k0 + c;
            const uint64_t db = db0 + (uint64_t)(((s * kCPS + c) * kBox) >> 4);
#pragma unroll
            for (int ks = 0; ks < kKChunk / 16; ++ks)   // K = 16: 8 TMEM columns of A, 32 B of W
              tc::umma_bf16_ta(d_tmem, tmem_base + (uint32_t)(kAcol + kc * 32 + ks * 8),
                               db + 2 * ks, kIdesc, (kc | ks) != 0 ? 1u : 0u);
          }
          tc::umma_commit(&b.bempty[s]);
        }
        if (ok) tc::umma_commit(&b.accfull[buf]);
      }
      // all issued MMAs complete before TMEM is released
      tc::umma_commit(b.mmadone);
      drain_bar(b.mmadone, 0);
    }
  } else {
    // ------------------------------------------------------ epilogue
    const int e = warp - 4;          // 0..7
    const int hs = e >> 2;           // column half of each tile
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;   // row within the M-tile
    const int n = r0 + row;          // global row b * gamma + j
    const bool valid = n < p.rows;
    const bool warp_rows = r0 + q * 32 < p.rows;   // does this warp hold any row?
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);

    // ---- A operand into TMEM: row n is E[prev_tok[n]] (zero when unbiased) ----
    // A 64-element K-chunk of a row is 128 contiguous bytes, 32 TMEM columns;
    // half hs stores the chunks bt = hs, hs + 2, ...
    {
      int tok = -1;
      if (valid && ((n % p.gamma) > 0 || p.bias_at_first)) {
        const int tk = p.prev_tok[n];
        if (tk < 0 || tk >= p.V)
          set_status(p.status, kErrArg);
        else
          tok = tk;
      }
      for (int bt = hs; bt < KC; bt += 2) {
        uint32_t v[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 w = make_uint4(0u, 0u, 0u, 0u);
          if (tok >= 0)
            w = __ldg(reinterpret_cast<const uint4*>(p.E + (size_t)tok * p.rank + bt * kKChunk +
                                                     c * 8));
          v[4 * c] = w.x;
          v[4 * c + 1] = w.y;
          v[4 * c + 2] = w.z;
          v[4 * c + 3] = w.w;
        }
        __syncwarp();
        tc::tmem_st_32x32b_x32(lane_base + (uint32_t)(kAcol + bt * 32), v);
      }
      tc::tmem_wait_st();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(b.aready);
    }

    // ---- per-row inputs of this pass ----
    int tgt = -1;
    float lq2 = 0.f, lp2 = 0.f;
    if (kPass == 1) {
      if (valid) tgt = p.target[n];
    } else {
      // pass 1's partials: wait until that grid has completed and its writes
      // are visible
      asm volatile("griddepcontrol.wait;" ::: "memory");
      if (valid) {
        Lse2 aq = lse2_empty(), ap = lse2_empty();
        for (int v = 0; v < p.n_vr; ++v) {
          const float4 f = __ldcg(&p.parts1[(size_t)v * p.rows_max + n]);
          aq = lse2_merge(aq, Lse2{f.x, f.y});
          ap = lse2_merge(ap, Lse2{f.z, f.w});
        }
        lq2 = aq.m + log2f(aq.s);
        lp2 = ap.m + log2f(ap.s);
      }
    }

    // ---- tiles ----
    Lse2 sq = lse2_empty(), sp = lse2_empty();   // pass 1
    float l1 = 0.f;                              // pass 2
    uint64_t* full = b.ufull + hs * kNU;
    uint64_t* empty = b.uempty + hs * kNU;
    const unsigned char* ring = sU + hs * kNU * kSlot;
    uint32_t uit = 0;
    for (int tt = 0; tt < nt; ++tt) {
      if (warp_aborted(abort_flag)) break;
      const int buf = tt % kNAcc;
      if (!warp_wait(&b.accfull[buf], (tt / kNAcc) & 1, abort_flag, p.status)) break;
      tc::tc_fence_after();
      const int vx = tile_of(tt) * kTileN + hs * kHalf;
      if (vx < p.V) {
        const int s = uit % kNU;
        if (!warp_wait(&full[s], (uit / kNU) & 1, abort_flag, p.status)) break;
        ++uit;
        const unsigned char* ubox = ring + s * kSlot;
        const unsigned char* pbox = ubox + kBox;
        // Both chunks go to registers first and the slot is released before
        // any arithmetic, so the producer can refill it while this tile is
        // computed: with two slots per half nearly the whole ring is in flight.
        uint4 uu[8], pp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uu[i] = box_chunk(ubox, row, i);
          pp[i] = box_chunk(pbox, row, i);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[s]);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint4* u = uu + 4 * c;
          const uint4* pw = pp + 4 * c;
          const int v0 = vx + c * 32;
          if (warp_rows && v0 < p.V) {
            uint32_t acc[32];
            tc::tmem_ld_32x32b_x32_wait(
                lane_base + (uint32_t)(kDcol + buf * kTileN + hs * kHalf + c * 32), acc);
            float xq[32], xp[32];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t uw[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
              const uint32_t pk[4] = {pw[i].x, pw[i].y, pw[i].z, pw[i].w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int x = 8 * i + 2 * k;
                add_bf16x2(uw[k], acc[x], acc[x + 1], xq[x], xq[x + 1]);
                xp[x] = bf16lo(pk[k]);
                xp[x + 1] = bf16hi(pk[k]);
              }
            }
            if (v0 + 32 > p.V) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (v0 + i >= p.V) {
                  xq[i] = -INFINITY;
                  xp[i] = -INFINITY;
                }
            }
            if (kPass == 1) {
              lse_fold32(sq, xq);
              lse_fold32(sp, xp);
              if ((unsigned)(tgt - v0) < 32u) {   // this thread's row has its target here
                float lt = xq[0];
#pragma unroll
                for (int i = 1; i < 32; ++i)
                  if (tgt - v0 == i) lt = xq[i];
                p.ltgt[n] = lt;
              }
            } else {
              l1 += l1_chunk32(xq, xp, lq2, lp2);
            }
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&b.accempty[buf]);
    }

    // ---- merge the two column halves of each row, publish the partial ----
    if (hs == 1) xch[row] = kPass == 1 ? make_float4(sq.m, sq.s, sp.m, sp.s)
                                       : make_float4(l1, 0.f, 0.f, 0.f);
    asm volatile("bar.sync 1, 256;" ::: "memory");   // the eight epilogue warps
    if (hs == 0 && valid) {
      const float4 o = xch[row];
      const size_t at = (size_t)vr * p.rows_max + n;
      if (kPass == 1) {
        const Lse2 mq = lse2_merge(sq, Lse2{o.x, o.y});
        const Lse2 mp = lse2_merge(sp, Lse2{o.z, o.w});
        p.parts1[at] = make_float4(mq.m, mq.s, mp.m, mp.s);
      } else {
        p.parts2[at] = l1 + o.x;
      }
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

constexpr int kFinThreads = 256;
constexpr int kFinWarps = kFinThreads / 32;

struct FinParams {
  const float4* parts1;
  const float* parts2;
  const float* ltgt;
  const int32_t* target;
  const float* conf_logit;
  float* row_out;            // [4][rows] (l1, accept, ce, bce) or nullptr
  float* losses;             // [4] (ce_loss, l1_loss, conf_loss, total)
  double* red;               // [gridDim.x][3] per-CTA sums
  unsigned int* ticket;      // zero between calls
  int* status;
  int rows, rows_max, n_vr, gamma, V;
  double w[kMaxGamma];       // normalised position weights (host, fp64)
  double ce_alpha, l1_alpha, conf_alpha;
};

// One thread per row: L1 = sum of the range partials; accept =
// clamp(1 - L1/2, 0, 1); CE = logsumexp(l) - l[target]; BCE with logits of
// the confidence against accept, max(z, 0) - z a + log(1 + e^-|z|).  The
// transcendentals are fp32 (their rounding is far below the fp32 inputs'
// own), the sums fp64.  Each CTA reduces its rows' w_j CE, w_j L1 and BCE;
// the last CTA to finish (a ticket) adds the CTA sums in CTA order, so the
// result does not depend on which CTA finishes last.
__global__ void __launch_bounds__(kFinThreads) loss_finalize_kernel(FinParams p) {
  __shared__ double red[3][kFinWarps];
  __shared__ int am_last;
  // launched behind pass 2 with a programmatic dependency: wait for its
  // partials (and, through it, pass 1's)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = blockIdx.x * kFinThreads + tid;
  double s_ce = 0.0, s_l1 = 0.0, s_bce = 0.0;
  if (n < p.rows) {
    Lse2 aq = lse2_empty();
    double l1 = 0.0;
    for (int v = 0; v < p.n_vr; ++v) {
      const float4 f = __ldcg(&p.parts1[(size_t)v * p.rows_max + n]);
      aq = lse2_merge(aq, Lse2{f.x, f.y});
      l1 += (double)__ldcg(&p.parts2[(size_t)v * p.rows_max + n]);
    }
    const int tg = p.target[n];
    float ce;
    if (tg < 0 || tg >= p.V) {
      set_status(p.status, kErrArg);
      ce = __int_as_float(0x7fc00000);   // NaN
    } else {
      ce = lse2_value(aq) - __ldcg(&p.ltgt[n]);
    }
    double a = 1.0 - 0.5 * l1;
    if (a < 0.0) a = 0.0;       // a NaN stays NaN and is reported below
    if (a > 1.0) a = 1.0;
    const float z = p.conf_logit[n];
    const float af = (float)a;
    const float bce = fmaxf(z, 0.f) - z * af + log1pf(expf(-fabsf(z)));
    const double w = p.w[n % p.gamma];
    s_ce = w * (double)ce;
    s_l1 = w * l1;
    s_bce = (double)bce;
    if (!isfinite(ce) || !isfinite(l1) || !isfinite(bce)) set_status(p.status, kErrNonfinite);
    if (p.row_out) {
      p.row_out[n] = (float)l1;
      p.row_out[(size_t)p.rows + n] = af;
      p.row_out[2 * (size_t)p.rows + n] = ce;
      p.row_out[3 * (size_t)p.rows + n] = bce;
    }
  }
  s_ce = warp_sum_f64(s_ce);
  s_l1 = warp_sum_f64(s_l1);
  s_bce = warp_sum_f64(s_bce);
  if (lane == 0) {
    red[0][warp] = s_ce;
    red[1][warp] = s_l1;
    red[2][warp] = s_bce;
  }
  __syncthreads();
  if (tid < 3) {
    double t = 0.0;
    for (int w = 0; w < kFinWarps; ++w) t += red[tid][w];
    p.red[blockIdx.x * 3 + tid] = t;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) am_last = (atomicAdd(p.ticket, 1u) == gridDim.x - 1) ? 1 : 0;
  __syncthreads();
  if (!am_last || tid != 0) return;
  __threadfence();
  double t[3] = {0.0, 0.0, 0.0};
  for (unsigned b = 0; b < gridDim.x; ++b)
    for (int i = 0; i < 3; ++i) t[i] += __ldcg(&p.red[b * 3 + i]);
  const double B = (double)(p.rows / p.gamma);
  const double ce_loss = t[0] / B, l1_loss = t[1] / B, conf_loss = t[2] / (double)p.rows;
  p.losses[0] = (float)ce_loss;
  p.losses[1] = (float)l1_loss;
  p.losses[2] = (float)conf_loss;
  p.losses[3] = (float)(p.ce_alpha * ce_loss + p.l1_alpha * l1_loss + p.conf_alpha * conf_loss);
  *p.ticket = 0u;   // ready for the next call (kernels on the stream run in order)
}

}  // namespace

// Vocabulary ranges per M-tile: the grid is M-tiles x ranges, one CTA per SM.
int loss_vranges(const Ctx& ctx, int rows) {
  const int MT = (rows + kTileM - 1) / kTileM;
  const int ntiles = (ctx.cfg.V + kTileN - 1) / kTileN;
  int n = ctx.num_sms / (MT > 0 ? MT : 1);
  if (n < 1) n = 1;
  if (n > ntiles) n = ntiles;
  return n;
}

cudaError_t launch_loss(const Ctx& ctx, const LossArgs& a, cudaStream_t s) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const int rows = a.B * a.gamma;
  const int MT = (rows + kTileM - 1) / kTileM;
  CUtensorMap tmW, tmU, tmP;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)a.rank, (cuuint64_t)a.V};
    const cuuint64_t strides[1] = {(cuuint64_t)a.rank * 2};
    const cuuint32_t box[2] = {kKChunk, (cuuint32_t)kTileN};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.W), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // U and P as [rows, V] matrices: [128 rows x 64 vocab] boxes; rows past the
  // batch and columns past V read as zero (and are masked or ignored).
  const void* srcs[2] = {a.U, a.P};
  CUtensorMap* maps[2] = {&tmU, &tmP};
  for (int i = 0; i < 2; ++i) {
    const cuuint64_t dims[2] = {(cuuint64_t)a.V, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)a.V * 2};
    const cuuint32_t box[2] = {kHalf, kTileM};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(srcs[i]), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(loss_tc_kernel<1>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kLossSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(loss_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kLossSmemBytes);
  if (e != cudaSuccess) return e;

  LossParams p{};
  p.E = static_cast<const __nv_bfloat16*>(a.E);
  p.prev_tok = a.prev_tok;
  p.target = a.target;
  p.parts1 = ctx.ws.loss_parts1;
  p.parts2 = ctx.ws.loss_parts2;
  p.ltgt = ctx.ws.loss_ltgt;
  p.status = ctx.ws.status;
  p.rows = rows;
  p.rows_max = ctx.cfg.R_max * ctx.cfg.gamma;
  p.V = a.V;
  p.rank = a.rank;
  p.gamma = a.gamma;
  p.bias_at_first = a.bias_at_first;
  p.n_vr = loss_vranges(ctx, rows);
  p.ntiles = (a.V + kTileN - 1) / kTileN;
  const int grid = MT * p.n_vr;

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kLThreads);
  cfg.dynamicSmemBytes = kLossSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  // pass 1 in plain stream order; pass 2 with a programmatic dependency on it
  cfg.numAttrs = 0;
  e = cudaLaunchKernelEx(&cfg, loss_tc_kernel<1>, tmW, tmU, tmP, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  count_launch(ctx);
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, loss_tc_kernel<2>, tmW, tmU, tmP, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  count_launch(ctx);

  FinParams f{};
  f.parts1 = ctx.ws.loss_parts1;
  f.parts2 = ctx.ws.loss_parts2;
  f.ltgt = ctx.ws.loss_ltgt;
  f.target = a.target;
  f.conf_logit = a.conf_logit;
  f.row_out = a.row_out;
  f.losses = a.losses;
  f.red = ctx.ws.loss_red;
  f.ticket = ctx.ws.tickets + 1;
  f.status = ctx.ws.status;
  f.rows = rows;
  f.rows_max = p.rows_max;
  f.n_vr = p.n_vr;
  f.gamma = a.gamma;
  f.V = a.V;
  double wsum = 0.0;
  for (int j = 0; j < a.gamma; ++j) wsum += exp(-(double)j / a.decay);
  for (int j = 0; j < a.gamma; ++j) f.w[j] = exp(-(double)j / a.decay) / wsum;
  f.ce_alpha = a.ce_alpha;
  f.l1_alpha = a.l1_alpha;
  f.conf_alpha = a.conf_alpha;
  cudaLaunchConfig_t fcfg = {};
  fcfg.gridDim = dim3((rows + kFinThreads - 1) / kFinThreads);
  fcfg.blockDim = dim3(kFinThreads);
  fcfg.stream = s;
  fcfg.attrs = attr;        // programmatic dependency on pass 2
  fcfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&fcfg, loss_finalize_kernel, f);
  if (e != cudaSuccess) return e;
  count_launch(ctx);
  return cudaGetLastError();
}

}  // namespace dsd
