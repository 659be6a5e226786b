// Warp-level tensor-core engine of dsd_propose (mma.sync m16n8k16, bf16 in,
// fp32 accumulate): one launch per draft step.
//
// Pages: "Qwen3.8-Flash-Next DSpark 训练实验", Baseline 架构 / Markov 顺序修正
// (m_i = W_1[t_{i-1}], b_i = W_2 m_i, l_i = l_i^0 + b_i, argmax over the full
// vocabulary); "DSpark notes" 2.3 (one lookup plus one low-rank projection);
// "DSpark 论文精读" 2.2 (x_j ~ Softmax(U_j + b)).
//
// Step j computes D[r, v] = sum_k M[r, k] W[v, k] for a 128-request M-tile
// (M = gathered rows E[x_{r, j-1}]) and the CTA's range of 128-wide
// vocabulary tiles.  Shared memory holds M (resident, 64 KB) and two W tiles
// (double-buffered with cp.async, 64 KB each); rows are 16-byte chunks
// XOR-swizzled by (row & 7) so that the ldmatrix row addresses of eight
// consecutive rows hit distinct banks.  Eight warps tile 128 x 128 as 2 (M) x
// 4 (N): each warp owns 64 requests x 32 vocabulary entries = 4 x 4
// m16n8 accumulators.  After each tile the accumulators plus U are folded
// into per-(thread, request-row) running base-2 log-sum-exp and argmax
// (greedy) or Gumbel-max (sampled) states; the biased logits never leave
// registers.  At the end the four threads of a quad and the four N-warps are
// merged and each request's partial is published (atomicMax of the packed
// key, one (m, s) partial per vocabulary range).
#include "dsd_common.cuh"

namespace dsd {

namespace {

constexpr int kMmaThreads = 256;
constexpr int kMT = 128;           // requests per CTA
constexpr int kNT = 128;           // vocabulary per tile
constexpr int kRowMax = 512;       // bytes of one K = 256 bf16 row
constexpr int kTileBytes = kNT * kRowMax;    // 64 KB
constexpr int kSmemMma = kMT * kRowMax + 2 * kTileBytes + 128;

struct MmaParams {
  const __nv_bfloat16* U;
  const __nv_bfloat16* E;
  const __nv_bfloat16* W;
  const int32_t* prev_tok;
  const uint32_t* req_id;
  unsigned long long* keys;   // [gamma][R_max]
  float2* parts;              // [gamma][n_part][R_max]
  int* status;
  int R, R_max, V, rank, gamma, j, bias_at_first, n_part, n_vr, ntiles, sampled;
  float inv_T;
  uint32_t k0, k1;
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of 16-byte chunk c of row r in a swizzled row-major tile.
__device__ __forceinline__ uint32_t swz(int r, int c, int row_bytes) {
  return (uint32_t)(r * row_bytes + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct RowSt {
  float m2, s, bz;
  uint32_t bv;
};

__device__ __forceinline__ void merge_into(RowSt& a, const RowSt& b) {
  const Lse2 l = lse2_merge(Lse2{a.m2, a.s}, Lse2{b.m2, b.s});
  a.m2 = l.m;
  a.s = l.s;
  if (b.bz > a.bz || (b.bz == a.bz && b.bv < a.bv)) {
    a.bz = b.bz;
    a.bv = b.bv;
  }
}

// Load one W tile (rows t*128 .. +127, all rank columns) into a buffer.
__device__ __forceinline__ void load_w_tile(const MmaParams& p, unsigned char* buf, int t, int tid) {
  const int cpr = p.rank / 8;                 // 16-byte chunks per row
  const int row_bytes = p.rank * 2;
  const uint32_t base = smem_addr(buf);
  for (int i = tid; i < kNT * cpr; i += kMmaThreads) {
    const int r = i / cpr, c = i - r * cpr;
    const int v = t * kNT + r;
    const bool ok = v < p.V;
    const __nv_bfloat16* src = p.W + (size_t)(ok ? v : 0) * p.rank + c * 8;
    cp_async16(base + swz(r, c, row_bytes), src, ok ? 16 : 0);
  }
}

__global__ void __launch_bounds__(kMmaThreads, 1) propose_mma_kernel(const MmaParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* sA = smem;
  unsigned char* sB0 = smem + kMT * kRowMax;
  unsigned char* sB1 = sB0 + kTileBytes;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp >> 2, wn = warp & 3;          // 2 x 4 warp grid
  const int mt = blockIdx.x / p.n_vr, vr = blockIdx.x - mt * p.n_vr;
  const int r_base = mt * kMT;
  const int t0 = (int)(((long long)vr * p.ntiles) / p.n_vr);
  const int t1 = (int)(((long long)(vr + 1) * p.ntiles) / p.n_vr);
  const int nt = t1 - t0;
  const int j = p.j;
  const int cpr = p.rank / 8;
  const int row_bytes = p.rank * 2;

  // first W tile in flight while the A operand is gathered
  if (nt > 0) load_w_tile(p, sB0, t0, tid);
  cp_async_commit();

  // ---- A: rows of E for the tokens of step j-1 (warp w: rows w*16 .. +15) ----
  {
    const bool biased = (j > 0) || p.bias_at_first;
    int my_tok = -1;
    if (lane < 16) {
      const int rr = r_base + warp * 16 + lane;
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
    uint4 v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int tok = __shfl_sync(0xffffffffu, my_tok, k);
      v[k] = make_uint4(0u, 0u, 0u, 0u);
      if (tok >= 0 && lane < cpr)
        v[k] = __ldcg(reinterpret_cast<const uint4*>(p.E + (size_t)tok * p.rank + lane * 8));
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int r = warp * 16 + k;
      if (lane < cpr) *reinterpret_cast<uint4*>(sA + swz(r, lane, row_bytes)) = v[k];
    }
  }

  // this thread's rows (8) and columns (8 per tile)
  RowSt st[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) st[i] = RowSt{-INFINITY, 0.f, -INFINITY, 0u};
  uint32_t rid[8];
  int rrow[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = r_base + wm * 64 + (i >> 1) * 16 + (lane >> 2) + (i & 1) * 8;
    rrow[i] = r;
    rid[i] = (r < p.R) ? (p.req_id ? p.req_id[r] : (uint32_t)r) : 0u;
  }
  const uint32_t a_base = smem_addr(sA);

  for (int tt = 0; tt < nt; ++tt) {
    const int t = t0 + tt;
    unsigned char* sB = (tt & 1) ? sB1 : sB0;
    if (tt + 1 < nt) load_w_tile(p, (tt & 1) ? sB0 : sB1, t + 1, tid);
    cp_async_commit();

    // U values of this tile: 8 rows x 4 column pairs
    const int vcol = t * kNT + wn * 32 + 2 * (lane & 3);
    uint32_t u[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int ni = 0; ni < 4; ++ni) {
        const int v = vcol + ni * 8;
        u[i][ni] = 0u;
        if (rrow[i] < p.R && v < p.V)
          u[i][ni] = __ldcs(reinterpret_cast<const unsigned int*>(
              p.U + ((size_t)rrow[i] * p.gamma + j) * p.V + v));
      }

    cp_async_wait<1>();
    __syncthreads();

    float acc[4][4][4];
#pragma unroll
    for (int mi = 0; mi < 4; ++mi)
#pragma unroll
      for (int ni = 0; ni < 4; ++ni)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mi][ni][e] = 0.f;

    const uint32_t b_base = smem_addr(sB);
    for (int ks = 0; ks < p.rank / 16; ++ks) {
      uint32_t af[4][4], bf[2][4];
#pragma unroll
      for (int mi = 0; mi < 4; ++mi) {
        const int r = wm * 64 + mi * 16 + (lane & 15);
        const int c = ks * 2 + (lane >> 4);
        ldsm_x4(a_base + swz(r, c, row_bytes), af[mi][0], af[mi][1], af[mi][2], af[mi][3]);
      }
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        const int n = wn * 32 + nb * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int c = ks * 2 + ((lane >> 3) & 1);
        ldsm_x4(b_base + swz(n, c, row_bytes), bf[nb][0], bf[nb][1], bf[nb][2], bf[nb][3]);
      }
#pragma unroll
      for (int mi = 0; mi < 4; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
          mma_bf16_16816(acc[mi][ni], af[mi], bf[ni >> 1][(ni & 1) * 2],
                         bf[ni >> 1][(ni & 1) * 2 + 1]);
    }

    // ---- fold the biased logits of this tile into the row states ----
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int mi = i >> 1, hf = i & 1;
      float xs[8];
#pragma unroll
      for (int ni = 0; ni < 4; ++ni) {
        xs[2 * ni] = acc[mi][ni][hf * 2] + bf16lo(u[i][ni]);
        xs[2 * ni + 1] = acc[mi][ni][hf * 2 + 1] + bf16hi(u[i][ni]);
      }
      if (t * kNT + kNT > p.V) {
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
          if (vcol + ni * 8 >= p.V) xs[2 * ni] = -INFINITY;
          if (vcol + ni * 8 + 1 >= p.V) xs[2 * ni + 1] = -INFINITY;
        }
      }
      if (p.sampled) {
#pragma unroll
        for (int e = 0; e < 8; ++e) xs[e] *= p.inv_T;
      }
      float cm = -INFINITY;
#pragma unroll
      for (int e = 0; e < 8; ++e) cm = fmaxf(cm, xs[e]);
      const float M = fmaxf(st[i].m2, cm * kLog2e);
      if (M != -INFINITY) {
        float sum = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) sum += exp2f(fmaf(xs[e], kLog2e, -M));
        st[i].s = st[i].s * exp2f(st[i].m2 - M) + sum;
        st[i].m2 = M;
      }
      if (!p.sampled) {
        if (cm > st[i].bz) {
          int best = 7;
#pragma unroll
          for (int e = 7; e >= 0; --e)
            if (xs[e] == cm) best = e;
          st[i].bz = cm;
          st[i].bv = (uint32_t)(vcol + (best >> 1) * 8 + (best & 1));
        }
      } else {
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
          const uint32_t v = (uint32_t)(vcol + ni * 8);
          const Philox4 ph = philox4x32_10(v >> 2, (uint32_t)j, rid[i], 0u, p.k0, p.k1);
          const float z0 = xs[2 * ni] + gumbel_from_word(philox_pick(ph, v & 3));
          const float z1 = xs[2 * ni + 1] + gumbel_from_word(philox_pick(ph, (v + 1) & 3));
          if (z0 > st[i].bz) {
            st[i].bz = z0;
            st[i].bv = v;
          }
          if (z1 > st[i].bz) {
            st[i].bz = z1;
            st[i].bv = v + 1;
          }
        }
      }
    }
    __syncthreads();   // every warp is done with this W buffer before it is refilled
  }
  cp_async_wait<0>();

  // ---- merge: the quad (same rows, other columns), then the four N-warps ----
#pragma unroll
  for (int i = 0; i < 8; ++i) {
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      RowSt other;
      other.m2 = __shfl_xor_sync(0xffffffffu, st[i].m2, o);
      other.s = __shfl_xor_sync(0xffffffffu, st[i].s, o);
      other.bz = __shfl_xor_sync(0xffffffffu, st[i].bz, o);
      other.bv = __shfl_xor_sync(0xffffffffu, st[i].bv, o);
      merge_into(st[i], other);
    }
  }
  __syncthreads();
  RowSt* scratch = reinterpret_cast<RowSt*>(sB0);   // [4 wn][128 rows]
  if ((lane & 3) == 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r_local = wm * 64 + (i >> 1) * 16 + (lane >> 2) + (i & 1) * 8;
      scratch[wn * kMT + r_local] = st[i];
    }
  }
  __syncthreads();
  if (tid < kMT) {
    RowSt m = scratch[tid];
    for (int w = 1; w < 4; ++w) merge_into(m, scratch[w * kMT + tid]);
    const int r = r_base + tid;
    if (r < p.R && nt > 0) {
      atomicMax(&p.keys[(size_t)j * p.R_max + r], make_key(m.bz, m.bv));
      p.parts[((size_t)j * p.n_part + vr) * p.R_max + r] = make_float2(m.m2, m.s);
    } else if (r < p.R) {
      p.parts[((size_t)j * p.n_part + vr) * p.R_max + r] = make_float2(-INFINITY, 0.f);
    }
  }
}

}  // namespace

int mma_vranges(const Ctx& ctx, int R) {
  const int MT = (R + kMT - 1) / kMT;
  const int ntiles = (ctx.cfg.V + kNT - 1) / kNT;
  int n = ctx.num_sms / (MT > 0 ? MT : 1);
  if (n < 1) n = 1;
  if (n > ntiles) n = ntiles;
  if (n > ctx.n_part) n = ctx.n_part;
  return n;
}

cudaError_t launch_propose_mma(const Ctx& ctx, const ProposeArgs& a, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(ctx.ws.keys, 0,
                                  sizeof(unsigned long long) * (size_t)a.gamma * ctx.cfg.R_max, s);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(propose_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemMma);
  if (e != cudaSuccess) return e;
  MmaParams p{};
  p.U = static_cast<const __nv_bfloat16*>(a.U);
  p.E = static_cast<const __nv_bfloat16*>(a.E);
  p.W = static_cast<const __nv_bfloat16*>(a.W);
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
  p.n_vr = mma_vranges(ctx, a.R);
  p.ntiles = (a.V + kNT - 1) / kNT;
  p.sampled = a.temperature > 0.f ? 1 : 0;
  p.inv_T = a.temperature > 0.f ? 1.f / a.temperature : 1.f;
  p.k0 = (uint32_t)(a.seed & 0xFFFFFFFFull);
  p.k1 = (uint32_t)(a.seed >> 32);
  const int MT = (a.R + kMT - 1) / kMT;
  for (int j = 0; j < a.gamma; ++j) {
    p.j = j;
    propose_mma_kernel<<<MT * p.n_vr, kMmaThreads, kSmemMma, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launch(ctx);
  }
  return cudaSuccess;
}

}  // namespace dsd
