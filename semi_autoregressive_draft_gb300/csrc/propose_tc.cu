// tcgen05 (5th-generation tensor core) engine of dsd_propose: one launch per
// draft step; CTA = one 128-request M-tile x a contiguous range of 128-wide
// vocabulary tiles, one CTA per SM.
//
// Pages: "Qwen3.8-Flash-Next DSpark 训练实验", Baseline 架构 / Markov 顺序修正
// (m_i = W_1[t_{i-1}], b_i = W_2 m_i, l_i = l_i^0 + b_i, greedy argmax over the
// full vocabulary); "DSpark notes" 2.3 (one lookup plus one low-rank
// projection per step); "DSpark 论文精读" 2.2 (x_j ~ Softmax(U_j + b)).
//
// Draft step j's bias projection for the whole batch is the GEMM
//     D[R, V] = M[R, r] * W[V, r]^T,    M[r_, :] = E[x_{r_, j-1}, :]
// with requests on the MMA's M dimension and the vocabulary on N.  The grid
// is (M-tiles) x (vocabulary ranges), so the CTAs of one range read the same
// W tiles at about the same time and all but the first read them from L2.
// Warp roles (12 warps):
//   warp 0      TMA producer of W tiles ([128 vocab x 64 K] boxes, 128-byte
//               swizzle, L2 evict-last: W stays resident across the steps),
//               two boxes per ring stage and barrier
//               into a 2-stage ring (64 KB)
//   warp 1      TMEM allocator and the single thread that issues tcgen05.mma
//               (M = 128, N = 128, K = 16 per instruction) into four fp32
//               accumulator buffers of 128 columns (512 columns)
//   warps 2, 3  TMA producers of U, one per 64-column half of each tile:
//               [128 requests x 64 vocab] boxes of the [V, gamma, R] view
//               (128-byte swizzle, evict-first: U is read once), each into its
//               own 3-slot ring
//   warps 4-11  epilogue, four warps (the four TMEM lane quarters) per column
//               half: first they gather the A operand (rows of E for the tokens
//               chosen at step j-1) into shared memory in the UMMA K-major
//               128-byte-swizzled layout; then thread = one request row and
//               64 columns per tile: tcgen05.ld brings 32 accumulator columns
//               at a time, U comes from shared memory, and the biased logits
//               are folded into a running base-2 log-sum-exp and an argmax
//               (greedy) or Gumbel-max (sampled) key; they never leave
//               registers.
//
// With at most 64 requests (one half-empty M-tile) rows 64..127 of A repeat
// rows 0..63, and the warps of lane quarters 2 and 3, which would otherwise
// hold no request, fold the second 32-column chunk of every 64-column half
// while quarters 0 and 1 fold the first: the tensor pipe computes each bias
// twice (it has the slack) and the per-thread epilogue work, the sampled
// path's Philox blocks included, halves.  The copies' states merge at the
// end through shared memory.
//
// Every mbarrier has exactly one consumer role that waits on each of its
// phases in order (a parity wait cannot tell phase k from phase k + 2, so no
// waiter may skip a phase).  That is why each column half has its own U ring
// and producer: with one ring shared by both halves, a group's consecutive
// waits on a slot would skip the other group's phase.
//
// At the end each CTA publishes per-request partials: atomicMax of the packed
// argmax key and an (m, s) log-sum-exp partial per vocabulary range.  The
// next step's launch reads the keys, so the kernel boundary is the batch-wide
// synchronisation between steps.  Every mbarrier wait is bounded: on time-out
// the kernel records DSD_ERR_TIMEOUT, stops issuing work, waits (bounded) for
// its own copies in flight, frees its TMEM and returns.
#include <stdio.h>
#include <stdlib.h>

#include <atomic>

#include "head_step.cuh"
#include "tc_common.cuh"

namespace dsd {

namespace {

constexpr int kTcThreads = 384;
constexpr int kTileN = 128;          // vocabulary rows per tile (UMMA N)
constexpr int kTileM = 128;          // requests per M-tile (UMMA M)
constexpr int kKChunk = 64;          // K elements per 128-byte swizzle row
constexpr int kMaxKC = 4;            // rank <= 256
constexpr int kBox = 16384;          // one [128 x 64] bf16 box (W or U)
constexpr int kCPS = 2;              // W boxes (K-chunks) per ring stage: one barrier each way
constexpr int kNB = 2;               // W ring stages
constexpr int kHalf = 64;            // vocabulary columns per U box (half a tile)
constexpr int kNU = 3;               // U ring slots per column half
constexpr int kNAcc = 4;             // accumulator buffers of kTileN columns
constexpr int kTmemCols = kNAcc * kTileN;
constexpr uint32_t kIdesc = tc::idesc_bf16_f32(kTileM, kTileN);

constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kMaxKC * kBox;            // 64 KB of A
constexpr int kOffU = kOffB + kNB * kCPS * kBox;        // + 64 KB of W
constexpr int kOffBar = kOffU + 2 * kNU * kBox;         // + 96 KB of U
// bfull, bempty, ufull[2], uempty[2], accfull, accempty, aready, mmadone
constexpr int kNumBars = 2 * kNB + 4 * kNU + 2 * kNAcc + 2;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 64 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
static_assert(kOffB % 1024 == 0 && kOffU % 1024 == 0, "swizzled boxes need aligned bases");
static_assert(kTmemCols == 512, "TMEM allocation is a power of two <= 512 columns");

#ifdef DSD_TC_CHECKS
// Self-checking build: an out-of-range index records a distinct status code
// (-100 - site) and the access is skipped instead of performed.
#define TC_CHECK(cond, site) (((cond)) ? true : (set_status(p.status, -100 - (site)), false))
#else
#define TC_CHECK(cond, site) true
#endif

constexpr int kStepAbort = kMaxGamma;    // abort word of a several-position launch
constexpr int kHeadSync = 32;            // + 2 j + phase: the head's step phases of position j
static_assert(kStepAbort < kHeadSync && kHeadSync + 2 * kMaxGamma <= kStepSyncWords,
              "step counters fit the workspace words");

struct TcParams {
  const __nv_bfloat16* E;
  const int32_t* prev_tok;
  const uint32_t* req_id;
  unsigned long long* keys;  // [gamma][R_max]
  float2* parts;             // [gamma][n_part][R_max]
  int* status;
  int j;                     // draft position of this launch (the first, if several)
  int j_end;                 // one past the last draft position of this launch
  unsigned int* step_sync;   // several positions per launch: [kMaxGamma] CTAs done with
                             // position j (zero before the launch); the last entry is the
                             // launch's abort word
  int R, R_max, V, rank, gamma, bias_at_first, n_part, n_vr, ntiles, sampled;
  int dup;                   // R <= 64: rows 64..127 repeat rows 0..63 and take the second
                             // 32-column chunk of every 64-column half
  const float* A;            // split mode: the head's representations [R, gamma, rank] f32
                             // (gated / RNN heads), or nullptr: act(E[x_{j-1}])
  int act;                   // split mode without A: the activation of the E rows
  float inv_T;
  uint32_t k0, k1;
  int head;                  // split mode in one launch: 1 gated head, 2 RNN head (their
                             // per-step work runs inside the launch), else 0
  HeadStepParams hs;         // the head's step arguments (head != 0)
  unsigned long long* cand_parts;   // candidate mode: [gamma][n_part][cand_R][kCandK] keys
  int cand_R;
};

struct Bars {
  uint64_t* bfull;      // [kNB]
  uint64_t* bempty;     // [kNB]
  uint64_t* ufull;      // [2][kNU]
  uint64_t* uempty;     // [2][kNU]
  uint64_t* accfull;    // [kNAcc]
  uint64_t* accempty;   // [kNAcc]
  uint64_t* aready;
  uint64_t* mmadone;
};

struct RowState {
  float m2, s, best_z;
  uint32_t best_v;
};

// x = u (bf16, widened exactly) + acc (fp32) for the two halves of one
// 32-bit word of U, one instruction each.
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

// Process N (16 or 32) consecutive columns of one request row: x = acc + u
// (fp32), masked beyond V; fold into the base-2 log-sum-exp and the argmax
// key.  The log-sum-exp state (m2, s) means sum = s * 2^m2.  Its reference
// m2 is only raised when the chunk maximum exceeds it by more than
// kLagBits, so the exponentials of a chunk do not wait for the chunk's
// maximum; pairs of columns go through the packed fp32x2 pipe and the sum is
// a tree.
template <int N>
__device__ __forceinline__ void foldN(RowState& st, const uint32_t (&acc)[N], const uint4* u,
                                      int v0, const TcParams& p, uint32_t rid, int j) {
  static_assert(N == 16 || N == 32, "16 or 32 columns");
  constexpr int NG = N / 4;          // groups of four columns
  float xs[N];
#pragma unroll
  for (int c = 0; c < N / 8; ++c) {
    const uint32_t w[4] = {u[c].x, u[c].y, u[c].z, u[c].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = c * 8 + 2 * e;
      add_bf16x2(w[e], acc[i], acc[i + 1], xs[i], xs[i + 1]);
    }
  }
  if (v0 + N > p.V) {
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (v0 + i >= p.V) xs[i] = -INFINITY;
  }
  if (p.sampled) {
    const uint64_t t2 = tc::pack2(p.inv_T, p.inv_T);
#pragma unroll
    for (int i = 0; i < N; i += 2) {
      const uint64_t x2 = tc::mul2(tc::pack2(xs[i], xs[i + 1]), t2);
      tc::unpack2(x2, xs[i], xs[i + 1]);
    }
  }
  // maxima of the groups of four, then of the chunk
  float gm[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g)
    gm[g] = fmaxf(tc::max3(xs[4 * g], xs[4 * g + 1], xs[4 * g + 2]), xs[4 * g + 3]);
  float cm = fmaxf(gm[0], gm[1]);
#pragma unroll
  for (int g = 2; g < NG; g += 2) cm = tc::max3(cm, gm[g], gm[g + 1]);
  const float cm2 = cm * kLog2e;
  if (cm2 > st.m2 + kLagBits) {       // rare after the first chunks
    st.s *= tc::ex2(st.m2 - cm2);     // 0 while the state is empty
    st.m2 = cm2;
  }
  if (st.m2 != -INFINITY) {
    const uint64_t l2 = tc::pack2(kLog2e, kLog2e);
    const uint64_t nm = tc::pack2(-st.m2, -st.m2);
    uint64_t e2[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      float a, b;
      tc::unpack2(tc::fma2(tc::pack2(xs[2 * i], xs[2 * i + 1]), l2, nm), a, b);
      e2[i] = tc::pack2(tc::ex2(a), tc::ex2(b));
    }
#pragma unroll
    for (int w = N / 4; w >= 1; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) e2[i] = tc::add2(e2[i], e2[i + w]);
    float slo, shi;
    tc::unpack2(e2[0], slo, shi);
    st.s += slo + shi;
  }
  if (!p.sampled) {
    if (cm > st.best_z) {
      // lowest index attaining the maximum: first group, then within it
      int g = NG - 1;
#pragma unroll
      for (int k = NG - 2; k >= 0; --k)
        if (gm[k] == cm) g = k;
      float a0 = xs[0], a1 = xs[1], a2 = xs[2];
#pragma unroll
      for (int k = 1; k < NG; ++k)
        if (g == k) {
          a0 = xs[4 * k];
          a1 = xs[4 * k + 1];
          a2 = xs[4 * k + 2];
        }
      const int idx = 4 * g + (a0 == cm ? 0 : a1 == cm ? 1 : a2 == cm ? 2 : 3);
      st.best_z = cm;
      st.best_v = (uint32_t)(v0 + idx);
    }
  } else {
    float zb = st.best_z;
    uint32_t vb = st.best_v;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const uint32_t v = (uint32_t)(v0 + 4 * g);
      const Philox4 ph = philox4x32_10(v >> 2, (uint32_t)j, rid, 0u, p.k0, p.k1);
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

// The sequential head's work for position j inside a one-launch proposal
// (split mode): every epilogue warp of the grid takes outputs (request r,
// two units k) in turn, with the routines of the standalone step kernels;
// then the CTAs meet at a counter so that every output is written before any
// CTA gathers it.  The RNN head has two such phases (the new state, then the
// output from it).  After a failure the warps still pass both named barriers
// of every phase.
template <int EW>
__device__ __forceinline__ void head_step_phases(const TcParams& p, int j, int e,
                                                 volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  const int nw = (int)gridDim.x * EW, gw = (int)blockIdx.x * EW + e;
  constexpr int NK = 2;                       // outputs per warp task (rank % 8 == 0)
  const int per_r = p.rank / NK;
  const int n_task = p.R * per_r;
  const int nph = p.head == 2 ? 2 : 1;
  for (int ph = 0; ph < nph; ++ph) {
    if (!warp_aborted(abort_flag)) {
      for (int task = gw; task < n_task; task += nw) {
        const int r = task / per_r, k0 = (task - r * per_r) * NK;
        if (p.head == 1)
          gate_outputs_warp<__nv_bfloat16, NK>(p.hs, j, r, k0);
        else if (ph == 0)
          rnn_state_warp<__nv_bfloat16, NK>(p.hs, j, r, k0);
        else
          rnn_out_warp<__nv_bfloat16, NK>(p.hs, j, r, k0);
      }
    }
    unsigned int* ctr = &p.step_sync[kHeadSync + 2 * j + ph];
    asm volatile("bar.sync 1, %0;" ::"n"(32 * EW) : "memory");   // this CTA's outputs written
    if (e == 0 && lane == 0) {
      __threadfence();
      atomicAdd(ctr, 1u);
      if (!*abort_flag &&
          !wait_count_gpu(ctr, gridDim.x, &p.step_sync[kStepAbort], abort_flag, p.status))
        *abort_flag = 1;
      if (*abort_flag) atomicExch(&p.step_sync[kStepAbort], 1u);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * EW) : "memory");
  }
}

// ---------------------------------------------------------------------------
// Candidate mode (the Markov top-16 candidate sets, at most 32 requests, the
// repeated-rows kernel): the U boxes hold 64 rows, and the rest of the U
// region holds per request row a sorted top-16 of packed (logit, token) keys
// of this CTA's columns (largest first, 0 = empty), the key of its 16th
// entry (the admission threshold) and one 16-key buffer per folding thread
// (4 column groups x 2 copies).  Each thread appends the keys of its tile's
// columns that beat the threshold; after the tile one warp per row inserts
// them into the list (warp-parallel insertion: a ballot of the entries above
// the key gives its place, the rest shift down one lane) and the threshold
// rises.  The lists go to the global parts at the end of each position.
constexpr int kCandRows = 32;                              // request rows (R <= 32)
constexpr int kCandSlots = 8;                              // folding threads per row
constexpr int kCandUBox = kBox / 2;                        // a U box of 64 rows
constexpr int kCandOffBuf = 2 * kNU * kCandUBox;           // within the U region
constexpr int kCandOffCnt = kCandOffBuf + kCandRows * kCandSlots * kCandK * 8;
constexpr int kCandOffList = kCandOffCnt + kCandRows * kCandSlots * 4;
constexpr int kCandOffTau = kCandOffList + kCandRows * kCandK * 8;
static_assert(kCandOffTau + kCandRows * 8 <= 2 * kNU * kBox, "candidate state fits the U region");

// Append this thread's keys of N consecutive columns (x = acc + U, the
// biased logits before any temperature) that beat the row's threshold.
template <int N>
__device__ __forceinline__ void cand_filter(const uint32_t (&acc)[N], const uint4* u, int v0,
                                            int V, unsigned long long tau,
                                            unsigned long long* buf, int& cnt) {
  const float tv = tau ? key_value(tau) : -INFINITY;   // an empty list admits every key
#pragma unroll
  for (int c = 0; c < N / 8; ++c) {
    const uint32_t w[4] = {u[c].x, u[c].y, u[c].z, u[c].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = c * 8 + 2 * e;
      float x0, x1;
      add_bf16x2(w[e], acc[i], acc[i + 1], x0, x1);
      // a key equal in value to the threshold may still beat it by index
      if (x0 >= tv && v0 + i < V) {
        const unsigned long long k = make_key(x0, (uint32_t)(v0 + i));
        if (k > tau) buf[cnt++] = k;
      }
      if (x1 >= tv && v0 + i + 1 < V) {
        const unsigned long long k = make_key(x1, (uint32_t)(v0 + i + 1));
        if (k > tau) buf[cnt++] = k;
      }
    }
  }
}

// One warp: merge the row's appended keys (kCandSlots buffers with counts
// cnt[]) into its sorted list, 32 keys at a time.  Every key is distinct (the
// token index is in its low bits) and 0 marks an empty entry, so a key's
// place in the merged list is the number of keys above it in the list and in
// the batch: lane l ranks the batch's key l, lanes 0..15 rank the list's
// entries, and every key with a place below 16 is written there.  Then the
// threshold (the 16th key, 0 while the list is not full).
__device__ __forceinline__ void cand_insert_row(unsigned long long* list, unsigned long long* tau,
                                                const unsigned long long* bufs, int* cnt) {
  const int lane = threadIdx.x & 31;
  int n[kCandSlots], pre[kCandSlots];
  int total = 0;
#pragma unroll
  for (int sl = 0; sl < kCandSlots; ++sl) {
    n[sl] = cnt[sl];
    pre[sl] = total;
    total += n[sl];
  }
  if (total == 0) return;
  for (int b0 = 0; b0 < total; b0 += 32) {
    const unsigned long long L = lane < kCandK ? list[lane] : 0ull;
    unsigned long long K = 0ull;
    const int f = b0 + lane;
    if (f < total) {
      // key f of the flattened buffers: slot q with pre[q] <= f, at f - pre[q]
      int adj = 0;
#pragma unroll
      for (int q = 1; q < kCandSlots; ++q)
        if (f >= pre[q]) adj = q * kCandK - pre[q];
      K = bufs[f + adj];
    }
    // the batch's keys sit in lanes 0 .. n_b - 1 (the shuffles bound the
    // merge, so only those lanes are visited)
    const int n_b = total - b0 < 32 ? total - b0 : 32;
    int rk = 0, rl = lane;   // list entries above list entry `lane`: lane
#pragma unroll
    for (int i = 0; i < kCandK; ++i) rk += __shfl_sync(0xffffffffu, L, i) > K ? 1 : 0;
    for (int i = 0; i < n_b; ++i) {
      const unsigned long long ki = __shfl_sync(0xffffffffu, K, i);
      rk += ki > K ? 1 : 0;
      rl += ki > L ? 1 : 0;
    }
    const int n_l = __popc(__ballot_sync(0xffffffffu, L != 0ull));
    const int n_k = n_b;
    const int n_u = n_l + n_k < kCandK ? n_l + n_k : kCandK;
    __syncwarp();
    if (L != 0ull && rl < kCandK) list[rl] = L;
    if (K != 0ull && rk < kCandK) list[rk] = K;
    if (lane >= n_u && lane < kCandK) list[lane] = 0ull;
    __syncwarp();
  }
  if (lane == 0) *tau = list[kCandK - 1];
  if (lane < kCandSlots) cnt[lane] = 0;
}

// EW epilogue warps (8, or 16 with setmaxnreg 56 / 104 as in the pair
// kernel): warp 4 + e folds column group e / 4 (EW / 4 groups of 128 / (EW/4)
// columns per tile) of TMEM lane quarter warp % 4.  DUP (at most 64
// requests): rows 64..127 of A repeat rows 0..63 and the two copies of a row
// fold the two halves of each group's columns.
template <int EW, bool DUP, bool SPLIT, bool CAND = false>
__global__ void __launch_bounds__(128 + 32 * EW, 1)
    propose_tc_kernel(const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmU, const TcParams p) {
  static_assert(!CAND || (DUP && !SPLIT && EW == 16), "candidates: the repeated-rows kernel");
  static_assert(!(DUP && SPLIT), "the split mode uses rows 64..127 of A for the low parts");
  constexpr int kRowsM = SPLIT ? 64 : kTileM;   // requests per M-tile
  constexpr int kUBytes = (SPLIT || CAND) ? kBox / 2 : kBox;   // one U box ([kRowsM x 64] bf16)
  constexpr int kUSlot = CAND ? kCandUBox : kBox;   // U ring slot stride
  constexpr int kGroups = EW / 4;               // column groups per tile
  constexpr int kGCols = kTileN / kGroups;      // columns of a group (64 or 32)
  constexpr int kFW = DUP ? kGCols / 2 : kGCols;   // columns one thread folds per tile
  constexpr int kChunk = kFW < 32 ? kFW : 32;   // columns per TMEM load and fold
  constexpr int kRowsPerWarp = kTileM / EW;     // A rows each epilogue warp gathers
  static_assert(EW == 8 || EW == 16, "8 or 16 epilogue warps");
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
  const int vr = blockIdx.x - mt * p.n_vr;
  const int r0 = mt * kRowsM;        // first request of this CTA's M-tile
  const int t0 = (int)(((long long)vr * p.ntiles) / p.n_vr);
  const int t1 = (int)(((long long)(vr + 1) * p.ntiles) / p.n_vr);
  const int nt = t1 - t0;

  // The next draft step's grid may start on SMs as this one's CTAs exit: it
  // initialises and prefetches W and U (inputs) while this step drains, and
  // waits for this step's argmax keys in griddepcontrol.wait below.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int i = 0; i < kNB; ++i) {
      tc::mbar_init(&b.bfull[i], 1);
      tc::mbar_init(&b.bempty[i], 1);
    }
    for (int i = 0; i < 2 * kNU; ++i) {
      tc::mbar_init(&b.ufull[i], 1);
      tc::mbar_init(&b.uempty[i], EW / 2);   // the warps that read a half
    }
    for (int i = 0; i < kNAcc; ++i) {
      tc::mbar_init(&b.accfull[i], 1);
      tc::mbar_init(&b.accempty[i], EW);
    }
    tc::mbar_init(b.aready, EW);
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

  if (warp < 4) {
  if constexpr (EW == 16) asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
  if (warp == 0) {
    // ------------------------------------------------------ W producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();
      uint32_t it = 0;
      for (int jj = p.j; jj < p.j_end; ++jj)     // the same W tiles at every position
      for (int t = t0; t < t1 && !*abort_flag; ++t)
        for (int k0 = 0; k0 < KC; k0 += kCPS, ++it) {
          const int s = it % kNB;
          const int nch = KC - k0 < kCPS ? KC - k0 : kCPS;
          if (!wait_bar(&b.bempty[s], ((it / kNB) & 1) ^ 1, abort_flag, p.status)) break;
          tc::mbar_arrive_expect_tx(&b.bfull[s], (uint32_t)(nch * kBox));
          for (int c = 0; c < nch; ++c)
            tc::tma_load_2d(sB + (s * kCPS + c) * kBox, &tmW, &b.bfull[s], (k0 + c) * kKChunk,
                            t * kTileN, pol);
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
    // ------------------------------------- U producer of column half hs
    const int hs = warp - 2;
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      uint64_t* full = b.ufull + hs * kNU;
      uint64_t* empty = b.uempty + hs * kNU;
      unsigned char* ring = sU + hs * kNU * kUSlot;
      uint32_t it = 0;
      for (int jj = p.j; jj < p.j_end; ++jj)
      for (int t = t0; t < t1 && !*abort_flag; ++t) {
        const int vx = t * kTileN + hs * kHalf;
        if (vx >= p.V) break;
        const int s = it % kNU;
        if (!wait_bar(&empty[s], ((it / kNU) & 1) ^ 1, abort_flag, p.status)) break;
        tc::mbar_arrive_expect_tx(&full[s], kUBytes);
        tc::tma_load_3d(ring + s * kUSlot, &tmU, &full[s], vx, jj, r0, pol);
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
      bool ok = true;
      // Descriptors of the first A box and the first W stage; the others
      // differ only in the start-address field, which counts 16-byte units.
      // Every operand lies inside this CTA's shared memory (< 2^18 bytes), so
      // adding an offset in those units never carries out of the field.
      const uint64_t da0 = tc::sdesc_kmajor_sw128(tc::smem_u32(sA));
      const uint64_t db0 = tc::sdesc_kmajor_sw128(tc::smem_u32(sB));
      uint32_t gt = 0;   // tiles of the launch so far (accumulator ring position)
      for (int jj = p.j; jj < p.j_end && ok; ++jj) {
      // A of position jj gathered (one phase of aready per position)
      ok = wait_bar(b.aready, (uint32_t)(jj - p.j) & 1u, abort_flag, p.status);
      tc::tc_fence_after();
      for (int tt = 0; tt < nt && ok; ++tt, ++gt) {
        const int buf = gt % kNAcc;
        ok = wait_bar(&b.accempty[buf], ((gt / kNAcc) & 1) ^ 1, abort_flag, p.status);
        if (!ok) break;
        tc::tc_fence_after();    // the epilogue's TMEM reads of this buffer are done
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * kTileN);
        for (int k0 = 0; k0 < KC; k0 += kCPS, ++bit) {
          const int s = bit % kNB;
          const int nch = KC - k0 < kCPS ? KC - k0 : kCPS;
          // TMA data: the mbarrier's completion makes it visible to the MMA
          ok = wait_bar(&b.bfull[s], (bit / kNB) & 1, abort_flag, p.status);
          if (!ok) break;
          for (int c = 0; c < nch; ++c) {
            const int kc = k0 + c;
            const uint64_t da = da0 + (uint64_t)((kc * kBox) >> 4);
            const uint64_t db = db0 + (uint64_t)(((s * kCPS + c) * kBox) >> 4);
#pragma unroll
            for (int ks = 0; ks < kKChunk / 16; ++ks) {   // K = 16 is 32 bytes = 2 units
              tc::umma_bf16(d_tmem, da + 2 * ks, db + 2 * ks, kIdesc, (kc | ks) != 0 ? 1u : 0u);
              // split: A's rows 64..127 (the low parts) start 8 KB into the
              // box; as rows 0..63 of a second MMA they add W lo to the same
              // accumulator rows (its rows 64..127 read past the box: unused)
              if constexpr (SPLIT)
                tc::umma_bf16(d_tmem, da + 512 + 2 * ks, db + 2 * ks, kIdesc, 1u);
            }
          }
          tc::umma_commit(&b.bempty[s]);
        }
        if (ok) tc::umma_commit(&b.accfull[buf]);
      }
      }
      // all issued MMAs complete before TMEM is released
      tc::umma_commit(b.mmadone);
      drain_bar(b.mmadone, 0);
    }
  }
  } else {
    // ------------------------------------------------------ epilogue
    if constexpr (EW == 16) asm volatile("setmaxnreg.inc.sync.aligned.u32 104;" ::: "memory");
    const int e = warp - 4;          // 0 .. EW - 1
    const int cg = e >> 2;           // column group of each tile
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;   // row within the M-tile
    // With dup, rows 64..127 hold the requests of rows 0..63 again (lane
    // quarters 2 and 3), and each copy folds its half of the group.
    const int rrow = DUP ? (row & 63) : row;   // the request's row (its U row)
    const int copy = DUP ? (q >> 1) : 0;       // the same for the whole warp
    const int cbase = cg * kGCols + copy * kFW;   // first column of this thread, in the tile
    const int hs = cbase / kHalf;    // the U box (column half) it reads
    const int r = r0 + rrow;
    // split: only rows 0..63 of the accumulator are requests
    const bool valid = r < p.R && (!SPLIT || row < kRowsM);
    const bool warp_rows = (!SPLIT || q < 2) && r0 + (DUP ? (q & 1) : q) * 32 < p.R;
    const uint32_t rid = valid ? (p.req_id ? p.req_id[r] : (uint32_t)r) : 0u;

    uint32_t gt = 0;    // tiles of the launch so far (accumulator ring position)
    uint32_t uit = 0;   // U boxes of the launch so far (U ring position)
    // After a failure (the CTA's abort flag) every warp still runs every
    // position's named barriers, with its waits failing at once, so that no
    // warp is left at a bar.sync.
    for (int j = p.j; j < p.j_end; ++j) {
    if (j == p.j) {
      // The keys of step j-1 come from the previous grid: wait until it has
      // completed and its writes are visible (a no-op without a programmatic
      // dependency).
      asm volatile("griddepcontrol.wait;" ::: "memory");
    } else {
      // every CTA of the launch has published position j - 1
      if (e == 0 && lane == 0 && !*abort_flag &&
          !wait_count_gpu(&p.step_sync[j - 1], gridDim.x, &p.step_sync[kStepAbort], abort_flag,
                          p.status))
        *abort_flag = 1;
      asm volatile("bar.sync 1, %0;" ::"n"(32 * EW) : "memory");
    }

    if constexpr (SPLIT) {
      if (p.head) head_step_phases<EW>(p, j, e, abort_flag);
    }
    if constexpr (SPLIT) {
      // ---- A operand, split: the fp32 representation a of each request
      // (the head's buffer, or act(E[x_{j-1}])) as hi = bf16(a) in row i and
      // lo = bf16(a - hi) in row 64 + i; |a - hi - lo| <= 2^-18 |a|.  This
      // warp fills rows e, e + EW, ... of the 64.
      constexpr int kSR = kRowsM / EW;
      const bool biased = (j > 0) || p.bias_at_first;
      int my_tok = -1;
      if (lane < kSR && !p.A) {
        const int rr = r0 + e + EW * lane;
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
      const int cpr = p.rank / 8;    // 8 elements per lane
      float a[kSR][8];
#pragma unroll
      for (int kk = 0; kk < kSR; ++kk) {
        const int rr = r0 + e + EW * kk;
        const int tok = __shfl_sync(0xffffffffu, my_tok, kk);
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) a[kk][q8] = 0.f;
        if (lane < cpr && biased && rr < p.R) {
          if (p.A) {
            const float4* src = reinterpret_cast<const float4*>(
                p.A + ((size_t)rr * p.gamma + j) * p.rank + lane * 8);
            const float4 x0 = __ldcg(src), x1 = __ldcg(src + 1);
            a[kk][0] = x0.x; a[kk][1] = x0.y; a[kk][2] = x0.z; a[kk][3] = x0.w;
            a[kk][4] = x1.x; a[kk][5] = x1.y; a[kk][6] = x1.z; a[kk][7] = x1.w;
          } else if (tok >= 0 &&
                     TC_CHECK((size_t)tok * p.rank + lane * 8 + 8 <= (size_t)p.V * p.rank, 2)) {
            const uint4 w = __ldcg(reinterpret_cast<const uint4*>(p.E + (size_t)tok * p.rank + lane * 8));
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
              a[kk][2 * q8] = act_apply(bf16lo(ws[q8]), p.act);
              a[kk][2 * q8 + 1] = act_apply(bf16hi(ws[q8]), p.act);
            }
          }
        }
      }
      if (lane < cpr) {
        const int kc = lane >> 3, c8 = lane & 7;
#pragma unroll
        for (int kk = 0; kk < kSR; ++kk) {
          const int ir = e + EW * kk;    // row 0..63; its low part goes to row 64 + ir
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            const __nv_bfloat16 h0 = __float2bfloat16_rn(a[kk][2 * q8]);
            const __nv_bfloat16 h1 = __float2bfloat16_rn(a[kk][2 * q8 + 1]);
            const __nv_bfloat16 l0 = __float2bfloat16_rn(a[kk][2 * q8] - __bfloat162float(h0));
            const __nv_bfloat16 l1 = __float2bfloat16_rn(a[kk][2 * q8 + 1] - __bfloat162float(h1));
            hw[q8] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
            lw[q8] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
          }
          const size_t off = (size_t)kc * kBox + ir * 128 + ((c8 ^ (ir & 7)) << 4);
          if (TC_CHECK(off + 64 * 128 + 16 <= (size_t)kMaxKC * kBox, 1)) {
            *reinterpret_cast<uint4*>(sA + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(sA + off + 64 * 128) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(b.aready);
    } else
    // ---- A operand: rows of E for the tokens of step j-1 ----
    // This warp fills rows e, e + EW, ...: lane k < kRowsPerWarp fetches the
    // token of row e + EW k, then the rows are copied into the 128-byte-
    // swizzled K-major layout of the UMMA descriptors.
    {
      const bool biased = (j > 0) || p.bias_at_first;
      int my_tok = -1;
      if (lane < kRowsPerWarp) {
        const int rr = r0 + (DUP ? ((e + EW * lane) & 63) : (e + EW * lane));
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
      uint4 v[kRowsPerWarp];
#pragma unroll
      for (int kk = 0; kk < kRowsPerWarp; ++kk) {
        const int tok = __shfl_sync(0xffffffffu, my_tok, kk);
        v[kk] = make_uint4(0u, 0u, 0u, 0u);
        if (tok >= 0 && lane < cpr &&
            TC_CHECK((size_t)tok * p.rank + lane * 8 + 8 <= (size_t)p.V * p.rank, 2))
          v[kk] = __ldcg(reinterpret_cast<const uint4*>(p.E + (size_t)tok * p.rank + lane * 8));
      }
      if (lane < cpr) {
        const int kc = lane >> 3, c8 = lane & 7;
#pragma unroll
        for (int kk = 0; kk < kRowsPerWarp; ++kk) {
          const int ir = e + EW * kk;
          const size_t off = (size_t)kc * kBox + ir * 128 + ((c8 ^ (ir & 7)) << 4);
          if (TC_CHECK(off + 16 <= (size_t)kMaxKC * kBox, 1))
            *reinterpret_cast<uint4*>(sA + off) = v[kk];
        }
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(b.aready);
    }

    // ---- tiles ----
    RowState st{-INFINITY, 0.f, -INFINITY, 0u};
    uint64_t* full = b.ufull + hs * kNU;
    uint64_t* empty = b.uempty + hs * kNU;
    const unsigned char* ring = sU + hs * kNU * kUSlot;
    const int c0 = (cbase - hs * kHalf) / 8;   // this thread's first 16-byte chunk of its U row
    // candidate mode: this thread's buffer, its row's list and threshold
    unsigned long long* c_list = reinterpret_cast<unsigned long long*>(sU + kCandOffList);
    unsigned long long* c_tau = reinterpret_cast<unsigned long long*>(sU + kCandOffTau);
    int* c_cnt = reinterpret_cast<int*>(sU + kCandOffCnt);
    unsigned long long* c_buf = reinterpret_cast<unsigned long long*>(sU + kCandOffBuf);
    const int c_slot = cg * 2 + copy;
    const bool c_row = CAND && valid && rrow < kCandRows;
    unsigned long long c_thr = 0ull;
    int c_n = 0;
    if constexpr (CAND) {
      // empty lists for position j: warp e clears rows e and e + 16
      for (int rr = e; rr < kCandRows; rr += EW) {
        if (lane < kCandK) c_list[rr * kCandK + lane] = 0ull;
        if (lane < kCandSlots) c_cnt[rr * kCandSlots + lane] = 0;
        if (lane == 0) c_tau[rr] = 0ull;
      }
      asm volatile("bar.sync 2, %0;" ::"n"(32 * EW) : "memory");
    }
    for (int tt = 0; tt < nt; ++tt, ++gt) {
      // A failed wait ends this warp's work; in candidate mode the warp still
      // passes every tile's named barriers.
      bool ok = !warp_aborted(abort_flag);
      const int t = t0 + tt;
      const int buf = gt % kNAcc;
      if (ok) ok = warp_wait(&b.accfull[buf], (gt / kNAcc) & 1, abort_flag, p.status);
      if (ok) {
        tc::tc_fence_after();
        const int vx = t * kTileN + hs * kHalf;
        if (vx < p.V) {
          const int s = uit % kNU;
          ok = warp_wait(&full[s], (uit / kNU) & 1, abort_flag, p.status);
          if (ok) {
            ++uit;
            // 128-byte swizzle: 16-byte chunk c of row `rrow` sits at chunk
            // c ^ (rrow & 7) of that row.
            uint4 u[kFW / 8];
            const unsigned char* urow = ring + s * kUSlot + rrow * 128;
            if (warp_rows) {
#pragma unroll
              for (int c = 0; c < kFW / 8; ++c)
                u[c] = *reinterpret_cast<const uint4*>(urow + (((c0 + c) ^ (rrow & 7)) << 4));
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&empty[s]);   // the slot's data is in registers
            __syncwarp();
            if (warp_rows) {
#pragma unroll
              for (int c = 0; c < kFW / kChunk; ++c) {
                const int v0 = t * kTileN + cbase + c * kChunk;
                if (v0 >= p.V) break;
                uint32_t acc[kChunk];
                tc::tmem_ld_wait<kChunk>(tmem_base + ((uint32_t)(q * 32) << 16) +
                                             (uint32_t)(buf * kTileN + cbase + c * kChunk),
                                         acc);
                foldN<kChunk>(st, acc, u + (kChunk / 8) * c, v0, p, rid, j);
                if constexpr (CAND) {
                  if (c_row)
                    cand_filter<kChunk>(acc, u + (kChunk / 8) * c, v0, p.V, c_thr,
                                        c_buf + (rrow * kCandSlots + c_slot) * kCandK, c_n);
                }
              }
            }
          }
        }
        if (ok) {
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&b.accempty[buf]);
        }
      }
      if constexpr (CAND) {
        // the tile's appends, then one warp per row inserts them
        if (c_row) c_cnt[rrow * kCandSlots + c_slot] = c_n;
        asm volatile("bar.sync 2, %0;" ::"n"(32 * EW) : "memory");
        for (int rr = e; rr < kCandRows; rr += EW)
          if (r0 + rr < p.R)
            cand_insert_row(c_list + rr * kCandK, c_tau + rr, c_buf + rr * kCandSlots * kCandK,
                            c_cnt + rr * kCandSlots);
        asm volatile("bar.sync 2, %0;" ::"n"(32 * EW) : "memory");
        c_n = 0;
        if (c_row) c_thr = c_tau[rrow];
      } else {
        if (!ok) break;
      }
    }
    if constexpr (CAND) {
      // this CTA's top-16 of every row for position j (the last tile's
      // insertions are complete: the loop ended on a named barrier)
      for (int rr = e; rr < kCandRows; rr += EW) {
        const int r_out = r0 + rr;
        if (r_out < p.R && r_out < p.cand_R && lane < kCandK && vr < p.n_part)
          p.cand_parts[(((size_t)j * p.n_part + vr) * p.cand_R + r_out) * kCandK + lane] =
              c_list[rr * kCandK + lane];
      }
    }

    // ---- merge the column groups (and with dup, the two copies) of each
    // row, publish step j's partial ----
    // The A region is free: the last accumulator barrier this warp waited on
    // was committed after every MMA that reads A, so they have all completed.
    RowState* xch = reinterpret_cast<RowState*>(sA);   // [kGroups][kTileM]
    RowState* xch2 = xch + kGroups * kTileM;           // dup: the second copy's merged state
    if (cg > 0) xch[(cg - 1) * kTileM + row] = st;
    asm volatile("bar.sync 1, %0;" ::"n"(32 * EW) : "memory");   // the epilogue warps
    if (cg == 0) {
#pragma unroll
      for (int k = 0; k < kGroups - 1; ++k) {
        const RowState o = xch[k * kTileM + row];
        const Lse2 l = lse2_merge(Lse2{st.m2, st.s}, Lse2{o.m2, o.s});
        st.m2 = l.m;
        st.s = l.s;
        if (o.best_z > st.best_z || (o.best_z == st.best_z && o.best_v < st.best_v)) {
          st.best_z = o.best_z;
          st.best_v = o.best_v;
        }
      }
      if (DUP && row >= 64) xch2[row - 64] = st;
    }
    if (DUP) {
      asm volatile("bar.sync 1, %0;" ::"n"(32 * EW) : "memory");
      if (cg == 0 && row < 64) {
        const RowState o = xch2[row];
        const Lse2 l = lse2_merge(Lse2{st.m2, st.s}, Lse2{o.m2, o.s});
        st.m2 = l.m;
        st.s = l.s;
        if (o.best_z > st.best_z || (o.best_z == st.best_z && o.best_v < st.best_v)) {
          st.best_z = o.best_z;
          st.best_v = o.best_v;
        }
      }
    }
    if (cg == 0 && (!DUP || row < 64) && valid && TC_CHECK(vr < p.n_part && r < p.R_max, 5)) {
      atomicMax(&p.keys[(size_t)j * p.R_max + r], make_key(st.best_z, st.best_v));
      p.parts[((size_t)j * p.n_part + vr) * p.R_max + r] = make_float2(st.m2, st.s);
    }
    if (j + 1 < p.j_end) {
      // position j published by this CTA (the merge's reads of the A region
      // done before the next gather writes it): one release arrival on the
      // launch's counter; an aborted CTA raises the launch's abort word
      asm volatile("bar.sync 1, %0;" ::"n"(32 * EW) : "memory");
      if (e == 0 && lane == 0) {
        __threadfence();
        atomicAdd(&p.step_sync[j], 1u);
        if (*abort_flag) atomicExch(&p.step_sync[kStepAbort], 1u);
      }
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

// ----------------------------------------------------------------------------
// Pair engine (an even number of M-tiles, e.g. R = 256): the two CTAs of a
// cluster are M-tiles 2i and 2i+1 of one vocabulary range, on two SMs.  Each
// CTA holds its own M-tile's A (gathered E rows) and U boxes as above, but
// only HALF of every W tile: vocabulary rows [t*128, t*128+64) in the first
// CTA of the pair, [t*128+64, t*128+128) in the second.  One thread of the
// first CTA issues tcgen05.mma.cta_group::2 with M = 256, N = 128: the
// tensor cores read A's rows 0..127 and B's first 64 rows from the first
// CTA's shared memory, A's rows 128..255 and B's last 64 rows from the
// second's, and write each CTA's 128 accumulator rows into its own TMEM.  So
// each SM takes in 32 KB of W per tile instead of 64 KB, and every W byte
// crosses L2 once per pair.  Each CTA's copies land in its own shared memory only.
//
// Barriers (per CTA; the first CTA's copies of aready, accempty and bfull
// collect both CTAs' arrivals):
//   bfull[s]    2 arrivals (each CTA's W producer: arrive.expect_tx of its own
//               bytes on the FIRST CTA's barrier) + the bytes of both halves,
//               whose TMA loads complete there (cta_group::2 form);
//   bempty[s]   1 arrival: the MMA thread's commit, issued to both CTAs'
//               barriers (two plain commits);
//   accfull[b]  1 arrival: commit to both CTAs after a tile's MMAs;
//   accempty[b] 16 arrivals (8 epilogue warps of each CTA) on the first CTA's;
//   aready      16 arrivals (A gathered in both CTAs) on the first CTA's;
//   ufull/uempty per CTA, as in the single-CTA kernel;
//   ugo         16 arrivals (this CTA's epilogue warps, first gather only).
// Every barrier still has one consumer role that waits on each of its phases
// in order.  Waits that see the peer's arrivals acquire at cluster scope.
constexpr int kPCPS = 4;                 // W half-boxes (K-chunks) per ring stage: a whole tile
constexpr int kPNB = 3;                  // W ring stages
constexpr int kPNU = 2;                  // U ring slots per column half
constexpr int kHalfBox = kBox / 2;       // [64 vocab x 64 K] bf16
constexpr uint32_t kIdescPair = tc::idesc_bf16_f32(2 * kTileM, kTileN);
constexpr int kPOffA = 0;
constexpr int kPOffB = kPOffA + kMaxKC * kBox;                // 64 KB of A
constexpr int kPOffU = kPOffB + kPNB * kPCPS * kHalfBox;      // + 96 KB of W halves
constexpr int kPOffBar = kPOffU + 2 * kPNU * kBox;            // + 64 KB of U
constexpr int kPNumBars = 2 * kPNB + 4 * kPNU + 2 * kNAcc + 3;
constexpr int kPSmemBytes = kPOffBar + kPNumBars * 8 + 64 + 1024;
static_assert(kPSmemBytes <= 232448, "shared memory budget of one CTA");
static_assert(kPOffB % 1024 == 0 && kPOffU % 1024 == 0 && kHalfBox % 1024 == 0,
              "swizzled boxes need aligned bases");

// EW epilogue warps per CTA: 8 (thread = one row, 64 columns of each tile)
// or 16 (32 columns each; the role warps hand registers to the epilogue with
// setmaxnreg).  Column group cq = (warp - 4) / 4 of a tile, lane quarter
// warp % 4.
template <int EW>
__global__ void __launch_bounds__(128 + 32 * EW, 1)
    propose_tc_pair_kernel(const __grid_constant__ CUtensorMap tmW,
                           const __grid_constant__ CUtensorMap tmU, const TcParams p) {
  constexpr int kGroups = EW / 4;             // column groups per tile
  constexpr int kGCols = kTileN / kGroups;    // columns per epilogue warp and tile
  constexpr int kGPerHalf = kGroups / 2;      // column groups per U box (half tile)
  constexpr int kRowsPerWarp = kTileM / EW;   // A rows each epilogue warp gathers
  static_assert(EW == 8 || EW == 16, "8 or 16 epilogue warps");
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  // the same offset in both CTAs (same kernel, same static shared memory), so
  // the MMA's descriptors address the peer's operands too
  unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  unsigned char* sA = smem + kPOffA;
  unsigned char* sB = smem + kPOffB;
  unsigned char* sU = smem + kPOffU;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPOffBar);
  Bars b;
  b.bfull = bars;
  b.bempty = b.bfull + kPNB;
  b.ufull = b.bempty + kPNB;
  b.uempty = b.ufull + 2 * kPNU;
  b.accfull = b.uempty + 2 * kPNU;
  b.accempty = b.accfull + kNAcc;
  b.aready = b.accempty + kNAcc;
  b.mmadone = b.aready + 1;
  uint64_t* ugo = b.mmadone + 1;   // this CTA's first A operand is gathered
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kPNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kPNumBars) + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int KC = p.rank / kKChunk;
  const uint32_t crank = tc::cluster_ctarank();      // 0: issues the MMAs
  const int cid = (int)(blockIdx.x >> 1);
  const int mt = 2 * (cid / p.n_vr) + (int)crank;
  const int vr = cid % p.n_vr;
  const int r0 = mt * kTileM;
  const int t0 = (int)(((long long)vr * p.ntiles) / p.n_vr);
  const int t1 = (int)(((long long)(vr + 1) * p.ntiles) / p.n_vr);
  const int nt = t1 - t0;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int i = 0; i < kPNB; ++i) {
      tc::mbar_init(&b.bfull[i], 2);
      tc::mbar_init(&b.bempty[i], 1);
    }
    for (int i = 0; i < 2 * kPNU; ++i) {
      tc::mbar_init(&b.ufull[i], 1);
      tc::mbar_init(&b.uempty[i], 4 * kGPerHalf);   // the warps that read a half
    }
    for (int i = 0; i < kNAcc; ++i) {
      tc::mbar_init(&b.accfull[i], 1);
      tc::mbar_init(&b.accempty[i], 2 * EW);
    }
    tc::mbar_init(b.aready, 2 * EW);
    tc::mbar_init(b.mmadone, 1);
    tc::mbar_init(ugo, EW);
    *abort_flag = 0;
    tc::mbar_fence_init();
    tc::fence_proxy_async_smem();
    tc::prefetch_tensormap(&tmW);
    tc::prefetch_tensormap(&tmU);
  }
  if (warp == 1) {
    __syncwarp();
    tc::tmem_alloc_pair(tmem_holder, kTmemCols);   // both CTAs, the same columns
    tc::tmem_relinquish_pair();
    tc::tc_fence_before();
  }
  __syncthreads();
  // the peer's copies, arrivals and commits may only target initialised barriers
  tc::cluster_sync();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // cluster addresses of the first CTA's collecting barriers
  const uint32_t bfull0 = tc::mapa(tc::smem_u32(b.bfull), 0);
  const uint32_t accempty0 = tc::mapa(tc::smem_u32(b.accempty), 0);
  const uint32_t aready0 = tc::mapa(tc::smem_u32(b.aready), 0);
  if (warp < 4) {
  // 16 epilogue warps: the role warpgroup (warps 0-3) gives registers to the
  // four epilogue warpgroups (within the 640 x 96 the CTA was launched with:
  // 128 x 56 + 512 x 104 <= 640 x 96)
  if constexpr (EW == 16) asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
  if (warp == 0) {
    // ------------------------------------- W producer: this CTA's half rows
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();
      uint32_t it = 0;
      for (int jj = p.j; jj < p.j_end; ++jj)     // the same W tiles at every position
      for (int t = t0; t < t1 && !*abort_flag; ++t)
        for (int k0 = 0; k0 < KC; k0 += kPCPS, ++it) {
          const int s = it % kPNB;
          const int nch = KC - k0 < kPCPS ? KC - k0 : kPCPS;
          if (!wait_bar_cl(&b.bempty[s], ((it / kPNB) & 1) ^ 1, abort_flag, p.status)) break;
          // relaxed: the bytes, not this thread's writes, complete the phase
          tc::mbar_arrive_expect_tx_cluster_relaxed(bfull0 + 8u * s, (uint32_t)(nch * kHalfBox));
          for (int c = 0; c < nch; ++c)
            tc::tma_load_2d_pair(sB + (s * kPCPS + c) * kHalfBox, &tmW, bfull0 + 8u * s,
                                 (k0 + c) * kKChunk, t * kTileN + (int)crank * (kTileN / 2), pol);
        }
      // Tail: the first CTA waits (bounded) for the last stages' copies of
      // both halves; each CTA waits for the MMA thread's release of its
      // stages (commit arrivals land asynchronously).
      if (crank == 0)
        for (uint32_t k = (it > kPNB ? it - kPNB : 0); k < it; ++k)
          drain_bar_cl(&b.bfull[k % kPNB], (k / kPNB) & 1);
      for (uint32_t k = (it > kPNB ? it - kPNB : 0); k < it; ++k)
        drain_bar_cl(&b.bempty[k % kPNB], (k / kPNB) & 1);
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------- U producer of column half hs
    const int hs = warp - 2;
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      uint64_t* full = b.ufull + hs * kPNU;
      uint64_t* empty = b.uempty + hs * kPNU;
      unsigned char* ring = sU + hs * kPNU * kBox;
      uint32_t it = 0;
      // the first U boxes wait for this CTA's first E-row gather, which would
      // otherwise queue behind them in DRAM (U is needed only after the first
      // MMA; W starts at once)
      wait_bar(ugo, 0, abort_flag, p.status);
      for (int jj = p.j; jj < p.j_end; ++jj)
      for (int t = t0; t < t1 && !*abort_flag; ++t) {
        const int vx = t * kTileN + hs * kHalf;
        if (vx >= p.V) break;
        const int s = it % kPNU;
        if (!wait_bar(&empty[s], ((it / kPNU) & 1) ^ 1, abort_flag, p.status)) break;
        tc::mbar_arrive_expect_tx(&full[s], kBox);
        tc::tma_load_3d(ring + s * kBox, &tmU, &full[s], vx, jj, r0, pol);
        ++it;
      }
      for (uint32_t k = (it > kPNU ? it - kPNU : 0); k < it; ++k)
        drain_bar(&full[k % kPNU], (k / kPNU) & 1);
      for (uint32_t k = (it > kPNU ? it - kPNU : 0); k < it; ++k)
        drain_bar(&empty[k % kPNU], (k / kPNU) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------- MMA issuer (first CTA only)
    if (lane == 0 && crank == 0) {
      uint32_t bit = 0;
      const uint32_t bempty_own = tc::smem_u32(b.bempty);
      const uint32_t bempty_peer = tc::mapa(bempty_own, 1);
      const uint32_t accfull_own = tc::smem_u32(b.accfull);
      const uint32_t accfull_peer = tc::mapa(accfull_own, 1);
      const uint64_t da0 = tc::sdesc_kmajor_sw128(tc::smem_u32(sA));
      const uint64_t db0 = tc::sdesc_kmajor_sw128(tc::smem_u32(sB));
      bool ok = true;
      uint32_t gt = 0;   // tiles of the launch so far (accumulator ring position)
      for (int jj = p.j; jj < p.j_end && ok; ++jj) {
      // A of position jj gathered in both CTAs (one phase of aready per position)
      ok = wait_bar_cl(b.aready, (uint32_t)(jj - p.j) & 1u, abort_flag, p.status);
      tc::tc_fence_after();
      for (int tt = 0; tt < nt && ok; ++tt, ++gt) {
        const int buf = gt % kNAcc;
        ok = wait_bar_cl(&b.accempty[buf], ((gt / kNAcc) & 1) ^ 1, abort_flag, p.status);
        if (!ok) break;
        tc::tc_fence_after();    // both CTAs' TMEM reads of this buffer are done
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * kTileN);
        for (int k0 = 0; k0 < KC; k0 += kPCPS, ++bit) {
          const int s = bit % kPNB;
          const int nch = KC - k0 < kPCPS ? KC - k0 : kPCPS;
          ok = wait_bar_cl(&b.bfull[s], (bit / kPNB) & 1, abort_flag, p.status);
          if (!ok) break;
          for (int c = 0; c < nch; ++c) {
            const int kc = k0 + c;
            const uint64_t da = da0 + (uint64_t)((kc * kBox) >> 4);
            const uint64_t db = db0 + (uint64_t)(((s * kPCPS + c) * kHalfBox) >> 4);
#pragma unroll
            for (int ks = 0; ks < kKChunk / 16; ++ks)
              tc::umma_bf16_pair(d_tmem, da + 2 * ks, db + 2 * ks, kIdescPair,
                                 (kc | ks) != 0 ? 1u : 0u);
          }
          tc::umma_commit_pair(bempty_own + 8u * s);     // the stage is free in both CTAs
          tc::umma_commit_pair(bempty_peer + 8u * s);
        }
        if (ok) {
          tc::umma_commit_pair(accfull_own + 8u * buf);
          tc::umma_commit_pair(accfull_peer + 8u * buf);
        }
      }
      }
      // all issued MMAs (which read both CTAs' shared memory and write both
      // TMEMs) complete before the pair passes the final cluster barrier
      tc::umma_commit_pair(tc::smem_u32(b.mmadone));
      drain_bar_cl(b.mmadone, 0);
    }
  }
  } else {
    // ------------------------------------------------------ epilogue
    if constexpr (EW == 16) asm volatile("setmaxnreg.inc.sync.aligned.u32 104;" ::: "memory");
    const int e = warp - 4;
    const int cq = e >> 2;           // column group of each tile
    const int hs = cq / kGPerHalf;   // U ring (column half) it reads
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int r = r0 + row;
    const bool valid = r < p.R;
    const bool warp_rows = r0 + q * 32 < p.R;
    const uint32_t rid = valid ? (p.req_id ? p.req_id[r] : (uint32_t)r) : 0u;

    uint32_t gt = 0;    // tiles of the launch so far (accumulator ring position)
    uint32_t uit = 0;   // U boxes of the launch so far (U ring position)
    // After a failure (the CTA's abort flag) every warp still runs every
    // position's named barriers, with its waits failing at once, so that no
    // warp is left at a bar.sync.
    for (int j = p.j; j < p.j_end; ++j) {
    if (j == p.j) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
    } else {
      // every CTA of the launch has published position j - 1
      if (e == 0 && lane == 0 && !*abort_flag &&
          !wait_count_gpu(&p.step_sync[j - 1], gridDim.x, &p.step_sync[kStepAbort], abort_flag,
                          p.status))
        *abort_flag = 1;
      asm volatile("bar.sync 1, %0;" ::"n"(32 * EW) : "memory");
    }

    // ---- A operand: rows of E for the tokens of step j-1 (this M-tile) ----
    // This warp fills rows e, e + EW, ...: lane k < kRowsPerWarp fetches the
    // token of row e + EW k, then the rows are copied into the 128-byte-
    // swizzled K-major layout of the UMMA descriptors.
    {
      const bool biased = (j > 0) || p.bias_at_first;
      int my_tok = -1;
      if (lane < kRowsPerWarp) {
        const int rr = r0 + e + EW * lane;
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
      const int cpr = p.rank / 8;
      uint4 v[kRowsPerWarp];
#pragma unroll
      for (int kk = 0; kk < kRowsPerWarp; ++kk) {
        const int tok = __shfl_sync(0xffffffffu, my_tok, kk);
        v[kk] = make_uint4(0u, 0u, 0u, 0u);
        if (tok >= 0 && lane < cpr &&
            TC_CHECK((size_t)tok * p.rank + lane * 8 + 8 <= (size_t)p.V * p.rank, 2))
          v[kk] = __ldcg(reinterpret_cast<const uint4*>(p.E + (size_t)tok * p.rank + lane * 8));
      }
      if (lane < cpr) {
        const int kc = lane >> 3, cc = lane & 7;
#pragma unroll
        for (int kk = 0; kk < kRowsPerWarp; ++kk) {
          const int ir = e + EW * kk;
          const size_t off = (size_t)kc * kBox + ir * 128 + ((cc ^ (ir & 7)) << 4);
          if (TC_CHECK(off + 16 <= (size_t)kMaxKC * kBox, 1))
            *reinterpret_cast<uint4*>(sA + off) = v[kk];
        }
      }
      tc::fence_proxy_async_smem();      // visible to the tensor cores of either SM
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_cluster(aready0);
      if (lane == 0 && j == p.j) tc::mbar_arrive(ugo);
    }

    // ---- tiles ----
    RowState st{-INFINITY, 0.f, -INFINITY, 0u};
    uint64_t* full = b.ufull + hs * kPNU;
    uint64_t* empty = b.uempty + hs * kPNU;
    const unsigned char* ring = sU + hs * kPNU * kBox;
    for (int tt = 0; tt < nt; ++tt, ++gt) {
      if (warp_aborted(abort_flag)) break;
      const int t = t0 + tt;
      const int buf = gt % kNAcc;
      if (!warp_wait_cl(&b.accfull[buf], (gt / kNAcc) & 1, abort_flag, p.status)) break;
      tc::tc_fence_after();
      const int vx = t * kTileN + hs * kHalf;        // first column of this warp's U box
      if (vx < p.V) {
        const int s = uit % kPNU;
        if (!warp_wait(&full[s], (uit / kPNU) & 1, abort_flag, p.status)) break;
        ++uit;
        // this warp's kGCols columns: 16-byte chunks c0 .. c0 + kGCols/8 - 1
        // of its row of the box (128-byte swizzle: chunk c at c ^ (row & 7))
        constexpr int kChunks = kGCols / 8;
        const int c0 = (cq % kGPerHalf) * kChunks;
        uint4 u[kChunks];
        const unsigned char* urow = ring + s * kBox + row * 128;
        if (warp_rows) {
#pragma unroll
          for (int c = 0; c < kChunks; ++c)
            u[c] = *reinterpret_cast<const uint4*>(urow + (((c0 + c) ^ (row & 7)) << 4));
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[s]);
        __syncwarp();
        if (warp_rows) {
#pragma unroll
          for (int c = 0; c < kGCols / 32; ++c) {
            const int v0 = vx + (c0 / 4 + c) * 32;
            if (v0 >= p.V) break;
            uint32_t acc[32];
            tc::tmem_ld_32x32b_x32_wait(tmem_base + ((uint32_t)(q * 32) << 16) +
                                            (uint32_t)(buf * kTileN + (v0 - t * kTileN)),
                                        acc);
            foldN<32>(st, acc, u + 4 * c, v0, p, rid, j);
          }
        }
      }
      // The TMEM reads are complete (tcgen05.wait::ld) and ordered by the
      // tcgen05 fence; the arrival publishes no memory writes, so it is
      // relaxed (a release at cluster scope costs a fence per tile and warp).
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_cluster_relaxed(accempty0 + 8u * buf);
    }

    // ---- merge the column groups of each row, publish step j's partial ----
    // The A region is free once this CTA's last accumulator wait has passed:
    // that commit followed every MMA that reads A.
    RowState* xch = reinterpret_cast<RowState*>(sA);   // [kGroups - 1][kTileM]
    if (cq > 0) xch[(cq - 1) * kTileM + row] = st;
    asm volatile("bar.sync 1, %0;" ::"n"(32 * EW) : "memory");   // the epilogue warps
    if (cq == 0) {
#pragma unroll
      for (int k = 0; k < kGroups - 1; ++k) {
        const RowState o = xch[k * kTileM + row];
        const Lse2 l = lse2_merge(Lse2{st.m2, st.s}, Lse2{o.m2, o.s});
        st.m2 = l.m;
        st.s = l.s;
        if (o.best_z > st.best_z || (o.best_z == st.best_z && o.best_v < st.best_v)) {
          st.best_z = o.best_z;
          st.best_v = o.best_v;
        }
      }
      if (valid && TC_CHECK(vr < p.n_part && r < p.R_max, 5)) {
        atomicMax(&p.keys[(size_t)j * p.R_max + r], make_key(st.best_z, st.best_v));
        p.parts[((size_t)j * p.n_part + vr) * p.R_max + r] = make_float2(st.m2, st.s);
      }
    }
    if (j + 1 < p.j_end) {
      // position j published by this CTA: one release arrival on the
      // launch's counter (an aborted CTA raises the launch's abort word)
      asm volatile("bar.sync 1, %0;" ::"n"(32 * EW) : "memory");
      if (e == 0 && lane == 0) {
        __threadfence();
        atomicAdd(&p.step_sync[j], 1u);
        if (*abort_flag) atomicExch(&p.step_sync[kStepAbort], 1u);
      }
    }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  // neither CTA leaves while the pair's MMAs, copies or arrivals may still
  // address its shared memory or TMEM
  tc::cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc::tc_fence_after();
    tc::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ----------------------------------------------------------------------------
// Residual pass of sampled verification on the tensor cores ("DeepSpec 训练
// 全流程详解" 4.4: after the first rejection at position k the next token is
// drawn from norm(max(0, p_k - q_k))).  For each request in the rejection
// list, q_k = softmax((U[r,k] + W E[x_{k-1}]) / T) is recomputed from its
// definition with the stored lse_q, p_k = softmax(P[r,k] / T) with the row
// pass's lse of P, and the draw is a Gumbel-max (Philox stream 2) over
// log(p - q) where p > q; the draw from p itself (the empty-residual
// fallback) and the two sums sum(p - q)+ and sum(p) are kept beside it.
//
// CTA = 64 rows of the rejection list (the list order is the row order) x a
// vocabulary range, 12 warps as in the propose kernel with 64 rows:
// A (the gathered E rows of x_{k-1}) holds rows 0..63 twice, so lane
// quarters 2 and 3 fold the second 32-column chunk of each 64-column half.
// The U and P rows of the listed (request, position) pairs are scattered in
// memory, so warps 2 and 3 fetch them as 1-D bulk copies (one per row and
// half tile, 16-byte aligned, a multiple of 16 bytes) into padded 144-byte
// row slots of a ring (the padding puts the rows read by a quarter warp in
// distinct banks).  W tiles and the MMA are as in the propose kernel.
// Outputs, as the CUDA-core residual pass: atomicMax of the residual key and
// of the fallback key per request, atomicAdd of the two sums.
constexpr int kRRows = 64;                       // list rows per CTA
constexpr int kRStride = 144;                    // bytes per row slot (128 + 16 of padding)
constexpr int kRArr = kRRows * kRStride;         // one array (U or P) of one slot
constexpr int kRSlot = 2 * kRArr;                // U rows, then P rows
constexpr int kRNU = 2;                          // slots per column half
constexpr int kROffA = 0;
constexpr int kROffB = kROffA + kMaxKC * kBox;               // 64 KB of A
constexpr int kROffU = kROffB + kNB * kCPS * kBox;           // + 64 KB of W
constexpr int kROffBar = kROffU + 2 * kRNU * kRSlot;         // + 72 KB of U and P rows
constexpr int kRNumBars = 2 * kNB + 4 * kRNU + 2 * kNAcc + 2;
constexpr int kRSmemBytes = kROffBar + kRNumBars * 8 + 64 + 1024;
static_assert(kRSmemBytes <= 232448, "shared memory budget of one CTA");
static_assert(kROffB % 1024 == 0 && kROffU % 1024 == 0 && kRStride % 16 == 0, "alignment");

struct ResParams {
  const __nv_bfloat16* E;
  const __nv_bfloat16* U;
  const __nv_bfloat16* P;
  const int32_t* prev_tok;
  const int32_t* tokens;
  const uint32_t* req_id;
  const float* lse_q;
  const int* rej_list;
  const int* rej_k;
  const float* rej_lseP;
  const unsigned int* n_rej;
  unsigned long long* res_keys;   // [2][R_max]: residual key, fallback key
  float* res_sums;                // [2][R_max]: sum (p - q)+, sum p
  int* status;
  int R, R_max, V, rank, gamma, bias_at_first, n_vr, ntiles;
  float inv_T;
  uint32_t k0, k1;
};

struct ResState {
  unsigned long long best, best2;   // residual key, fallback key
  float fsum, fsum2;
};

// A thread's running state of the two draws inside the tile loop, each an
// exponential race: the Gumbel-max draw argmax_v ln w_v - ln(-ln u_v) is
// argmax_v w_v / t_v with t_v = -ln u_v, so the residual draw compares
// (p - q) / t and the fallback draw p / t, by cross products, without
// logarithms of the weights; the winner (w, t) becomes the key
// ln w - ln t = ln w + g after the tile loop (race_keys).
struct ResRace {
  float rb, tb;     // residual: best p - q and its t (rb = 0: none yet)
  float fb, tfb;    // fallback: best p and its t
  uint32_t vb, vfb;
  float fsum, fsum2;
};

// WC consecutive columns of one row (a multiple of 4): x = acc + U, then
// p and q from their base-2 logits on the special-function unit (2^x), the
// residual p - q, one Philox block per four columns for the races' t, and
// the sums of (p - q)+ and of p.  uw / pw: the row's U and P values, two
// bf16 per word.  p - q carries the error of the logits it comes from
// (about 1e-6 of p), as the logarithm of the difference did.
template <int WC>
__device__ __forceinline__ void fold_res(ResRace& st, const uint32_t (&acc)[WC],
                                         const uint32_t* uw, const uint32_t* pw, int v0,
                                         const ResParams& p, uint32_t rid, uint32_t pos, float lq,
                                         float lp) {
  const float sT = p.inv_T * kLog2e, lq2 = lq * kLog2e, lp2 = lp * kLog2e;
#pragma unroll
  for (int g = 0; g < WC / 4; ++g) {
    const uint32_t v = (uint32_t)(v0 + 4 * g);
    if (v >= (uint32_t)p.V) break;   // V % 8 == 0: groups of four are all in or all out
    float xs[4], ps[4];
    add_bf16x2(uw[2 * g], acc[4 * g], acc[4 * g + 1], xs[0], xs[1]);
    add_bf16x2(uw[2 * g + 1], acc[4 * g + 2], acc[4 * g + 3], xs[2], xs[3]);
    ps[0] = bf16lo(pw[2 * g]);
    ps[1] = bf16hi(pw[2 * g]);
    ps[2] = bf16lo(pw[2 * g + 1]);
    ps[3] = bf16hi(pw[2 * g + 1]);
    const Philox4 ph = philox4x32_10(v >> 2, pos, rid, 2u, p.k0, p.k1);
    const uint32_t words[4] = {ph.x, ph.y, ph.z, ph.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float pv = tc::ex2(fmaf(ps[e], sT, -lp2));   // p
      const float qv = tc::ex2(fmaf(xs[e], sT, -lq2));   // q
      const float t = neg_ln_uniform(words[e]);
      const float r = pv - qv;
      if (r > 0.f) {
        st.fsum += r;
        if (r * st.tb > st.rb * t) {
          st.rb = r;
          st.tb = t;
          st.vb = v + e;
        }
      }
      if (pv * st.tfb > st.fb * t) {
        st.fb = pv;
        st.tfb = t;
        st.vfb = v + e;
      }
      st.fsum2 += pv;
    }
  }
}

// The races' winners as packed keys (0: no entry with a positive weight).
__device__ __forceinline__ ResState race_keys(const ResRace& st) {
  ResState o;
  o.best = st.rb > 0.f ? make_key((lg2_approx(st.rb) - lg2_approx(st.tb)) * kLn2, st.vb) : 0ull;
  o.best2 = st.fb > 0.f ? make_key((lg2_approx(st.fb) - lg2_approx(st.tfb)) * kLn2, st.vfb) : 0ull;
  o.fsum = st.fsum;
  o.fsum2 = st.fsum2;
  return o;
}

// One tile of one thread of the residual epilogue: its WC columns starting at
// column `col` of the tile (TMEM lane = its row of A).
template <int WC>
__device__ __forceinline__ void res_tile(ResRace& st, uint32_t tmem_addr,
                                         const unsigned char* urow, const unsigned char* prow,
                                         bool active, int v0, const ResParams& p, uint32_t rid,
                                         uint32_t pos, float lq, float lp) {
  uint32_t uw[WC / 2], pw[WC / 2];
  if (active) {
    static_assert(WC == 16 || WC == 32, "a copy folds 16 or 32 columns of a half");
    {
#pragma unroll
      for (int c = 0; c < WC / 8; ++c) {
        const uint4 a = *reinterpret_cast<const uint4*>(urow + 16 * c);
        const uint4 b = *reinterpret_cast<const uint4*>(prow + 16 * c);
        uw[4 * c] = a.x; uw[4 * c + 1] = a.y; uw[4 * c + 2] = a.z; uw[4 * c + 3] = a.w;
        pw[4 * c] = b.x; pw[4 * c + 1] = b.y; pw[4 * c + 2] = b.z; pw[4 * c + 3] = b.w;
      }
    }
  }
  // `active` differs between lanes: the warp reconverges before the
  // warp-wide (.sync.aligned) tensor-memory load
  __syncwarp();
  uint32_t acc[WC];
  tc::tmem_ld_wait<WC>(tmem_addr, acc);
  if (active) fold_res<WC>(st, acc, uw, pw, v0, p, rid, pos, lq, lp);
}

__global__ void __launch_bounds__(kTcThreads, 1)
    residual_tc_kernel(const __grid_constant__ CUtensorMap tmW, const ResParams p) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ int s_req[kRRows];
  __shared__ int s_pos[kRRows];
  __shared__ int s_tok[kRRows];     // x_{k-1}, or -1 without a bias

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = blockIdx.x / p.n_vr;
  const int vr = blockIdx.x - mt * p.n_vr;
  const int n_rej = min((int)*p.n_rej, p.R);
  const int li0 = mt * kRRows;
  if (li0 >= n_rej) return;          // the whole CTA, before any barrier or TMEM
  const int nvalid = min(kRRows, n_rej - li0);

  const uint32_t raw = tc::smem_u32(smem_raw);
  unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  unsigned char* sA = smem + kROffA;
  unsigned char* sB = smem + kROffB;
  unsigned char* sU = smem + kROffU;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kROffBar);
  Bars b;
  b.bfull = bars;
  b.bempty = b.bfull + kNB;
  b.ufull = b.bempty + kNB;
  b.uempty = b.ufull + 2 * kRNU;
  b.accfull = b.uempty + 2 * kRNU;
  b.accempty = b.accfull + kNAcc;
  b.aready = b.accempty + kNAcc;
  b.mmadone = b.aready + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kRNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kRNumBars) + 1;

  const int KC = p.rank / kKChunk;
  const int t0 = (int)(((long long)vr * p.ntiles) / p.n_vr);
  const int t1 = (int)(((long long)(vr + 1) * p.ntiles) / p.n_vr);
  const int nt = t1 - t0;

  if (tid < kRRows) {
    int req = 0, pos = 0, tok = -1;
    if (tid < nvalid) {
      req = p.rej_list[li0 + tid];
      if (req < 0 || req >= p.R) {
        set_status(p.status, kErrArg);
        req = 0;
      }
      pos = p.rej_k[req];
      if (pos < 0 || pos >= p.gamma) {
        set_status(p.status, kErrArg);
        pos = 0;
      }
      if (pos > 0 || p.bias_at_first) {
        tok = pos == 0 ? p.prev_tok[req] : p.tokens[(size_t)req * p.gamma + pos - 1];
        if (tok < 0 || tok >= p.V) {
          set_status(p.status, kErrArg);
          tok = 0;
        }
      }
    }
    s_req[tid] = req;
    s_pos[tid] = pos;
    s_tok[tid] = tok;
  }
  if (tid == 0) {
    for (int i = 0; i < kNB; ++i) {
      tc::mbar_init(&b.bfull[i], 1);
      tc::mbar_init(&b.bempty[i], 1);
    }
    for (int i = 0; i < 2 * kRNU; ++i) {
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
        for (int k0 = 0; k0 < KC; k0 += kCPS, ++it) {
          const int s = it % kNB;
          const int nch = KC - k0 < kCPS ? KC - k0 : kCPS;
          if (!wait_bar(&b.bempty[s], ((it / kNB) & 1) ^ 1, abort_flag, p.status)) break;
          tc::mbar_arrive_expect_tx(&b.bfull[s], (uint32_t)(nch * kBox));
          for (int c = 0; c < nch; ++c)
            tc::tma_load_2d(sB + (s * kCPS + c) * kBox, &tmW, &b.bfull[s], (k0 + c) * kKChunk,
                            t * kTileN, pol);
        }
      for (uint32_t k = (it > kNB ? it - kNB : 0); k < it; ++k)
        drain_bar(&b.bfull[k % kNB], (k / kNB) & 1);
      for (uint32_t k = (it > kNB ? it - kNB : 0); k < it; ++k)
        drain_bar(&b.bempty[k % kNB], (k / kNB) & 1);
    }
  } else if (warp == 2 || warp == 3) {
    // ---------------------- U and P rows of column half hs: bulk copies per row
    const int hs = warp - 2;
    const uint64_t pol = policy_evict_first();
    uint64_t* full = b.ufull + hs * kRNU;
    uint64_t* empty = b.uempty + hs * kRNU;
    unsigned char* ring = sU + hs * kRNU * kRSlot;
    // this lane's rows i = lane and lane + 32: the start of their U and P rows
    const __nv_bfloat16* usrc[2];
    const __nv_bfloat16* psrc[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = lane + 32 * h;
      const int req = s_req[i], pos = s_pos[i];
      usrc[h] = p.U + ((size_t)req * p.gamma + pos) * p.V;
      psrc[h] = p.P + ((size_t)req * (p.gamma + 1) + pos) * p.V;
    }
    uint32_t it = 0;
    for (int t = t0; t < t1; ++t) {
      if (warp_aborted(abort_flag)) break;
      const int vx = t * kTileN + hs * kHalf;
      if (vx >= p.V) break;
      const uint32_t bytes = (uint32_t)(min(kHalf, p.V - vx) * 2);   // a multiple of 16 (V % 8 == 0)
      const int s = it % kRNU;
      if (!warp_wait(&empty[s], ((it / kRNU) & 1) ^ 1, abort_flag, p.status)) break;
      if (lane == 0) tc::mbar_arrive_expect_tx(&full[s], (uint32_t)nvalid * 2u * bytes);
      __syncwarp();
      unsigned char* slot = ring + s * kRSlot;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        if (i < nvalid && TC_CHECK(kRArr + i * kRStride + (int)bytes <= kRSlot, 6)) {
          tc::bulk_load(slot + i * kRStride, usrc[h] + vx, bytes, &full[s], pol);
          tc::bulk_load(slot + kRArr + i * kRStride, psrc[h] + vx, bytes, &full[s], pol);
        }
      }
      ++it;
    }
    if (lane == 0) {
      for (uint32_t k = (it > kRNU ? it - kRNU : 0); k < it; ++k)
        drain_bar(&full[k % kRNU], (k / kRNU) & 1);
      for (uint32_t k = (it > kRNU ? it - kRNU : 0); k < it; ++k)
        drain_bar(&empty[k % kRNU], (k / kRNU) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t bit = 0;
      bool ok = wait_bar(b.aready, 0, abort_flag, p.status);
      tc::tc_fence_after();
      const uint64_t da0 = tc::sdesc_kmajor_sw128(tc::smem_u32(sA));
      const uint64_t db0 = tc::sdesc_kmajor_sw128(tc::smem_u32(sB));
      for (int tt = 0; tt < nt && ok; ++tt) {
        const int buf = tt % kNAcc;
        ok = wait_bar(&b.accempty[buf], ((tt / kNAcc) & 1) ^ 1, abort_flag, p.status);
        if (!ok) break;
        tc::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * kTileN);
        for (int k0 = 0; k0 < KC; k0 += kCPS, ++bit) {
          const int s = bit % kNB;
          const int nch = KC - k0 < kCPS ? KC - k0 : kCPS;
          ok = wait_bar(&b.bfull[s], (bit / kNB) & 1, abort_flag, p.status);
          if (!ok) break;
          for (int c = 0; c < nch; ++c) {
            const int kc = k0 + c;
            const uint64_t da = da0 + (uint64_t)((kc * kBox) >> 4);
            const uint64_t db = db0 + (uint64_t)(((s * kCPS + c) * kBox) >> 4);
#pragma unroll
            for (int ks = 0; ks < kKChunk / 16; ++ks)
              tc::umma_bf16(d_tmem, da + 2 * ks, db + 2 * ks, kIdesc, (kc | ks) != 0 ? 1u : 0u);
          }
          tc::umma_commit(&b.bempty[s]);
        }
        if (ok) tc::umma_commit(&b.accfull[buf]);
      }
      tc::umma_commit(b.mmadone);
      drain_bar(b.mmadone, 0);
    }
  } else {
    // ------------------------------------------------------ epilogue
    // A holds the list rows 128 / nrep times (nrep = 32 or 64): row i of A is
    // list row i % nrep, and its copy i / nrep folds nrep / 2 columns of each
    // 64-column half.  A copy spans whole lane quarters, so the copy index is
    // the same for every lane of a warp: a tensor-memory load addresses the
    // same columns for all 32 lanes of the warp.
    const int e = warp - 4;          // 0..7
    const int hs = e >> 2;           // column half of each tile
    const int q = warp & 3;          // TMEM lane quarter
    const int row = q * 32 + lane;   // row of A / TMEM lane
    const int nrep = nvalid <= 32 ? 32 : 64;
    const int lrow = row & (nrep - 1);     // the list row it holds
    const int copy = row / nrep;
    const int wc = nrep / 2;               // columns per copy and half
    const bool valid = lrow < nvalid;
    const int req = s_req[lrow];
    const uint32_t pos = (uint32_t)s_pos[lrow];
    const uint32_t rid = valid ? (p.req_id ? p.req_id[req] : (uint32_t)req) : 0u;
    const float lq = valid ? p.lse_q[(size_t)req * p.gamma + pos] : 0.f;
    const float lp = valid ? p.rej_lseP[req] : 0.f;
    if (valid && (!isfinite(lq) || !isfinite(lp))) set_status(p.status, kErrNonfinite);

    // ---- A operand: rows of E for x_{k-1} of each listed request ----
    {
      int my_tok = -1;
      if (lane < 16) my_tok = s_tok[(e + 8 * lane) & (nrep - 1)];
      const int cpr = p.rank / 8;
      uint4 v[16];
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const int tok = __shfl_sync(0xffffffffu, my_tok, kk);
        v[kk] = make_uint4(0u, 0u, 0u, 0u);
        if (tok >= 0 && lane < cpr &&
            TC_CHECK((size_t)tok * p.rank + lane * 8 + 8 <= (size_t)p.V * p.rank, 2))
          v[kk] = __ldcg(reinterpret_cast<const uint4*>(p.E + (size_t)tok * p.rank + lane * 8));
      }
      if (lane < cpr) {
        const int kc = lane >> 3, c8 = lane & 7;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const int ir = e + 8 * kk;
          const size_t off = (size_t)kc * kBox + ir * 128 + ((c8 ^ (ir & 7)) << 4);
          if (TC_CHECK(off + 16 <= (size_t)kMaxKC * kBox, 1))
            *reinterpret_cast<uint4*>(sA + off) = v[kk];
        }
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(b.aready);
    }

    ResRace st{0.f, 1.f, 0.f, 1.f, 0u, 0u, 0.f, 0.f};
    uint64_t* full = b.ufull + hs * kRNU;
    uint64_t* empty = b.uempty + hs * kRNU;
    const unsigned char* ring = sU + hs * kRNU * kRSlot;
    uint32_t uit = 0;
    for (int tt = 0; tt < nt; ++tt) {
      if (warp_aborted(abort_flag)) break;
      const int t = t0 + tt;
      const int buf = tt % kNAcc;
      if (!warp_wait(&b.accfull[buf], (tt / kNAcc) & 1, abort_flag, p.status)) break;
      tc::tc_fence_after();
      const int vx = t * kTileN + hs * kHalf;
      if (vx < p.V) {
        const int s = uit % kRNU;
        if (!warp_wait(&full[s], (uit / kRNU) & 1, abort_flag, p.status)) break;
        ++uit;
        const int v0 = vx + copy * wc;
        const bool active = valid && v0 < p.V;
        const unsigned char* urow = ring + s * kRSlot + lrow * kRStride + copy * wc * 2;
        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) +
                               (uint32_t)(buf * kTileN + hs * kHalf + copy * wc);
        // the tensor-memory load is warp-wide (every lane takes part); the
        // width is the same for the whole CTA
        if (wc == 16)
          res_tile<16>(st, taddr, urow, urow + kRArr, active, v0, p, rid, pos, lq, lp);
        else
          res_tile<32>(st, taddr, urow, urow + kRArr, active, v0, p, rid, pos, lq, lp);
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[s]);   // this warp's reads of the slot are done
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&b.accempty[buf]);
    }

    // ---- merge the 2 x 128 / nrep partial states of each list row ----
    // The A region is free: the last accumulator wait followed every MMA.
    ResState* xch = reinterpret_cast<ResState*>(sA);   // [2][kTileM]
    xch[hs * kTileM + row] = race_keys(st);
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (hs == 0 && row < nvalid && TC_CHECK(req < p.R_max, 5)) {
      ResState m{0ull, 0ull, 0.f, 0.f};
      for (int h = 0; h < 2; ++h)
        for (int c = 0; c < kTileM / nrep; ++c) {
          const ResState o = xch[h * kTileM + c * nrep + row];
          m.best = o.best > m.best ? o.best : m.best;
          m.best2 = o.best2 > m.best2 ? o.best2 : m.best2;
          m.fsum += o.fsum;
          m.fsum2 += o.fsum2;
        }
      if (m.best) atomicMax(&p.res_keys[req], m.best);
      if (m.best2) atomicMax(&p.res_keys[p.R_max + req], m.best2);
      atomicAdd(&p.res_sums[req], m.fsum);
      atomicAdd(&p.res_sums[p.R_max + req], m.fsum2);
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

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

int tc_supported(const Ctx& ctx, char* why, size_t why_len) {
  if (ctx.cfg.dtype != 1) {
    snprintf(why, why_len, "tcgen05 engine needs bf16 tables");
    return 0;
  }
  if (ctx.cfg.rank % kKChunk != 0 || ctx.cfg.rank > kMaxKC * kKChunk) {
    snprintf(why, why_len, "tcgen05 engine needs a Markov rank that is a multiple of 64, <= 256");
    return 0;
  }
  if (ctx.cfg.act != kActNone && ctx.cfg.act != kActSilu) {
    snprintf(why, why_len, "tcgen05 engine: unknown activation");
    return 0;
  }
  if (!tensor_map_encoder()) {
    snprintf(why, why_len, "cuTensorMapEncodeTiled is not available from the driver");
    return 0;
  }
  int smem = 0;
  cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, ctx.cfg.device);
  const int need = kSmemBytes > kPSmemBytes ? kSmemBytes : kPSmemBytes;
  if (smem < need) {
    snprintf(why, why_len, "device lacks %d bytes of shared memory per block", need);
    return 0;
  }
  return 1;
}

// The split mode (the Markov representation is not a bf16 row of E: an
// activation, or the gated / RNN head's fp32 representation) runs M-tiles of
// 64 requests with A's rows 64..127 holding the low parts.
static bool use_split(const Ctx& ctx, const ProposeArgs& a) {
  return a.act != kActNone || a.gate_h != nullptr;
}

// Vocabulary ranges per M-tile: the grid is M-tiles x ranges, one CTA per SM.
int tc_vranges_rows(const Ctx& ctx, int R, int rows_per_tile) {
  const int MT = (R + rows_per_tile - 1) / rows_per_tile;
  const int ntiles = (ctx.cfg.V + kTileN - 1) / kTileN;
  int n = ctx.num_sms / (MT > 0 ? MT : 1);
  if (n < 1) n = 1;
  if (n > ntiles) n = ntiles;
  if (n > ctx.n_part) n = ctx.n_part;
  return n;
}
int tc_vranges(const Ctx& ctx, int R) { return tc_vranges_rows(ctx, R, kTileM); }
int tc_vranges_split(const Ctx& ctx, int R) { return tc_vranges_rows(ctx, R, 64); }
// The partial slots a propose call on this engine fills (the finalize's n_used).
int tc_parts_used(const Ctx& ctx, const ProposeArgs& a) {
  return use_split(ctx, a) ? tc_vranges_split(ctx, a.R) : tc_vranges(ctx, a.R);
}

// An even number of M-tiles runs on CTA pairs (propose_tc_pair_kernel).
constexpr int kPairEpiWarps = 16;
constexpr int kSingleEpiWarps = 16;
static bool use_pair(int R) {
  const int MT = (R + kTileM - 1) / kTileM;
  return MT >= 2 && MT % 2 == 0;
}

// The single launch is cooperative unless DSD_PROPOSE_COOPERATIVE=0: ncu
// cannot replay a cooperative launch (the driver reports LaunchFailed), so
// profiling runs set it to 0 and time the same kernel launched without the
// attribute.  Read once.
static bool cooperative_launches() {
  static const bool on = [] {
    const char* v = getenv("DSD_PROPOSE_COOPERATIVE");
    return !(v && v[0] == '0');
  }();
  return on;
}

// Whether every CTA (or cluster) of a launch can be resident at once, one
// CTA per SM: the condition for running all draft steps in one cooperative
// launch, whose CTAs wait for one another between steps.  Asked once per
// kernel, device and grid.
template <auto Kernel>
static bool grid_resident(const Ctx& ctx, const cudaLaunchConfig_t& cfg, bool cluster) {
  // cache word: 1 (valid) | ok << 1 | grid << 2 | device << 34
  static std::atomic<unsigned long long> cache{0ull};
  const unsigned long long key =
      ((unsigned long long)(unsigned)ctx.cfg.device << 34) | ((unsigned long long)cfg.gridDim.x << 2);
  const unsigned long long c = cache.load(std::memory_order_relaxed);
  if ((c & 1ull) && (c & ~3ull) == key) return (c & 2ull) != 0;
  int n = 0;
  cudaError_t e;
  unsigned long long fits = 0;
  if (cluster) {
    cudaLaunchConfig_t q = cfg;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = 2;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    q.attrs = &at;
    q.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&n, Kernel, &q);
    fits = 2ull * (unsigned)n;
  } else {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, Kernel, (int)cfg.blockDim.x,
                                                      cfg.dynamicSmemBytes);
    fits = (unsigned long long)(unsigned)n * (unsigned)ctx.num_sms;
  }
  if (e != cudaSuccess) cudaGetLastError();   // unknown: one launch per step
  const bool ok = e == cudaSuccess && fits >= cfg.gridDim.x;
  cache.store(key | 1ull | (ok ? 2ull : 0ull), std::memory_order_relaxed);
  return ok;
}

cudaError_t launch_propose_tc(const Ctx& ctx, const ProposeArgs& a, cudaStream_t s) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const bool split = use_split(ctx, a);
  const bool pair = !split && use_pair(a.R);
  const int rows_m = split ? 64 : kTileM;   // requests per M-tile
  // candidate sets (at most 32 requests, no activation): the repeated-rows
  // kernel with 64-row U boxes
  const bool cand = a.cand_tok != nullptr;
  if (cand && (split || a.R > kCandRows)) return cudaErrorInvalidValue;
  const int u_rows = cand ? 64 : rows_m;   // rows of a U box
  CUtensorMap tmW, tmU;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)a.rank, (cuuint64_t)a.V};
    const cuuint64_t strides[1] = {(cuuint64_t)a.rank * 2};
    // a CTA of a pair loads half of each tile's vocabulary rows
    const cuuint32_t box[2] = {kKChunk, (cuuint32_t)(pair ? kTileN / 2 : kTileN)};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.W), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)a.V, (cuuint64_t)a.gamma, (cuuint64_t)a.R};
    const cuuint64_t strides[2] = {(cuuint64_t)a.V * 2, (cuuint64_t)a.V * 2 * a.gamma};
    const cuuint32_t box[3] = {kHalf, 1, (cuuint32_t)u_rows};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&tmU, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.U), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // the keys and, right after them, the position counters of a
  // several-position launch
  cudaError_t e = cudaMemsetAsync(ctx.ws.keys, 0,
                                  sizeof(unsigned long long) * (size_t)ctx.cfg.gamma * ctx.cfg.R_max +
                                      sizeof(unsigned int) * kStepSyncWords,
                                  s);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(propose_tc_kernel<kSingleEpiWarps, false, false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(propose_tc_kernel<kSingleEpiWarps, true, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(propose_tc_kernel<kSingleEpiWarps, true, false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(propose_tc_kernel<kSingleEpiWarps, false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(propose_tc_pair_kernel<kPairEpiWarps>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmemBytes);
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
  p.step_sync = ctx.ws.step_sync;
  p.n_vr = split ? tc_vranges_split(ctx, a.R) : tc_vranges(ctx, a.R);
  p.dup = !split && a.R <= kTileM / 2 ? 1 : 0;
  p.cand_parts = cand ? ctx.ws.cand_parts : nullptr;
  p.cand_R = ctx.cfg.R_max < kCandMaxR ? ctx.cfg.R_max : kCandMaxR;
  p.A = a.gate_h ? a.gated_rep : nullptr;
  p.act = a.act;
  const int grid = ((a.R + rows_m - 1) / rows_m) * p.n_vr;
  if (a.gate_h) {   // gated or RNN head: the hidden-state parts of every position, once
    e = a.rnn_W ? launch_rnn_h(ctx, a, s) : launch_gate_h(ctx, a, s);
    if (e != cudaSuccess) return e;
  }

  // The next step's A operand needs every CTA's argmax.  A grid that fits on
  // the device at once runs all draft steps in one launch, the CTAs meeting
  // at a counter per position (p.step_sync); otherwise (or with a head
  // kernel between the steps) one launch per step, steps after the first
  // launched with a programmatic dependency on the previous step (see
  // griddepcontrol in the kernel).
  // The first launch follows the memset of the keys in plain stream order.
  // Pairs: clusters of two CTAs, block 2 c + m = M-tile 2 (c / n_vr) + m of
  // vocabulary range c % n_vr.
  cudaLaunchAttribute cluster_attr, coop_attr, pdl_attr;
  cluster_attr.id = cudaLaunchAttributeClusterDimension;
  cluster_attr.val.clusterDim.x = pair ? 2 : 1;
  cluster_attr.val.clusterDim.y = 1;
  cluster_attr.val.clusterDim.z = 1;
  // a launch whose CTAs wait for one another is cooperative: it starts only
  // when every CTA can be resident, also beside other work on the device
  coop_attr.id = cudaLaunchAttributeCooperative;
  coop_attr.val.cooperative = 1;
  pdl_attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl_attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchAttribute attr[3];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(128 + 32 * (pair ? kPairEpiWarps : kSingleEpiWarps));
  cfg.dynamicSmemBytes = pair ? kPSmemBytes : kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  // all steps in one launch (with a gated or RNN head, the split kernel runs
  // the head's step work itself)
  bool whole = false;
  if (a.gamma > 1 && (!a.gate_h || split))
    whole = pair    ? grid_resident<propose_tc_pair_kernel<kPairEpiWarps>>(ctx, cfg, true)
            : cand  ? grid_resident<propose_tc_kernel<kSingleEpiWarps, true, false, true>>(ctx, cfg, false)
            : split ? grid_resident<propose_tc_kernel<kSingleEpiWarps, false, true>>(ctx, cfg, false)
            : p.dup ? grid_resident<propose_tc_kernel<kSingleEpiWarps, true, false>>(ctx, cfg, false)
                    : grid_resident<propose_tc_kernel<kSingleEpiWarps, false, false>>(ctx, cfg, false);
  if (whole && a.gate_h) {
    p.head = a.rnn_W ? 2 : 1;
    p.hs = head_step_params(ctx, a);
  }
  for (int j = 0; j < a.gamma; j = p.j_end) {
    p.j = j;
    p.j_end = whole ? a.gamma : j + 1;
    if (a.gate_h && !whole) {   // this step's representation from the tokens of the last
      e = a.rnn_W ? launch_rnn_step(ctx, a, j, s) : launch_gate_step(ctx, a, j, s);
      if (e != cudaSuccess) return e;
    }
    // a head kernel in between: plain stream order
    int na = 0;
    if (pair) attr[na++] = cluster_attr;
    if (whole) {
      if (cooperative_launches()) attr[na++] = coop_attr;
    } else if (j > 0 && !a.gate_h) {
      attr[na++] = pdl_attr;
    }
    cfg.numAttrs = (unsigned)na;
    e = pair    ? cudaLaunchKernelEx(&cfg, propose_tc_pair_kernel<kPairEpiWarps>, tmW, tmU, p)
        : cand  ? cudaLaunchKernelEx(&cfg, propose_tc_kernel<kSingleEpiWarps, true, false, true>, tmW, tmU, p)
        : split ? cudaLaunchKernelEx(&cfg, propose_tc_kernel<kSingleEpiWarps, false, true>, tmW, tmU, p)
        : p.dup ? cudaLaunchKernelEx(&cfg, propose_tc_kernel<kSingleEpiWarps, true, false>, tmW, tmU, p)
                : cudaLaunchKernelEx(&cfg, propose_tc_kernel<kSingleEpiWarps, false, false>, tmW, tmU, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launch(ctx);
  }
  return cudaSuccess;
}

// The residual pass of sampled verification on the tensor cores (same
// configurations as the propose engine: bf16 tables, no activation, rank a
// multiple of 64 <= 256).  The grid covers every list row the batch could
// need (ceil(R / 64) row blocks x vocabulary ranges); blocks past the
// device-side list length return at once.
cudaError_t launch_residual_tc(const Ctx& ctx, const VerifyArgs& a, cudaStream_t s) {
  if (a.R <= 0) return cudaSuccess;
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap tmW;
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
  cudaError_t e = cudaFuncSetAttribute(residual_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmemBytes);
  if (e != cudaSuccess) return e;
  ResParams p{};
  p.E = static_cast<const __nv_bfloat16*>(a.E);
  p.U = static_cast<const __nv_bfloat16*>(a.U);
  p.P = static_cast<const __nv_bfloat16*>(a.P);
  p.prev_tok = a.prev_tok;
  p.tokens = a.tokens;
  p.req_id = a.req_id;
  p.lse_q = a.lse_q;
  p.rej_list = ctx.ws.rej_list;
  p.rej_k = ctx.ws.rej_k;
  p.rej_lseP = ctx.ws.rej_lseP;
  p.n_rej = ctx.ws.counters + 1;
  p.res_keys = ctx.ws.res_keys;
  p.res_sums = ctx.ws.res_sums;
  p.status = ctx.ws.status;
  p.R = a.R;
  p.R_max = ctx.cfg.R_max;
  p.V = a.V;
  p.rank = a.rank;
  p.gamma = a.gamma;
  p.bias_at_first = a.bias_at_first;
  p.ntiles = (a.V + kTileN - 1) / kTileN;
  p.inv_T = 1.f / a.temperature;
  p.k0 = (uint32_t)(a.seed & 0xFFFFFFFFull);
  p.k1 = (uint32_t)(a.seed >> 32);
  const int MT = (a.R + kRRows - 1) / kRRows;
  int n_vr = ctx.num_sms / MT;
  if (n_vr < 1) n_vr = 1;
  if (n_vr > p.ntiles) n_vr = p.ntiles;
  p.n_vr = n_vr;
  residual_tc_kernel<<<MT * n_vr, kTcThreads, kRSmemBytes, s>>>(tmW, p);
  count_launch(ctx);
  return cudaGetLastError();
}

}  // namespace dsd
