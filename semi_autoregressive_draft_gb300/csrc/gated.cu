// Gated Markov head and RNN head, the sequential heads that read the
// backbone's hidden state.
//
// Gated Markov head ("DSpark 论文精读" 2.3, GatedMarkovHead):
//     m_j = act(E[x_{j-1}]),  g_j = sigmoid(W_g [h_j; m_j]),  b_j = W (g_j * m_j)
// W_g is [rank, H + rank], its hidden-state columns first.
//
// The gate's argument splits into a part that does not depend on the drafted
// tokens, W_g[:, :H] h_j, and one that does, W_g[:, H:] m_j.  The first is
// one dense product for all positions of the batch before the sequential
// stage (gate_h_kernel, [R gamma, H] x [H, rank] on CUDA cores, 64 x 64
// output tiles, split over H into partials); the second is a [rank, rank]
// matrix-vector product per request at each draft step (gate_step_kernel,
// one CTA per request and 8 gate outputs, one warp per output row,
// 16-byte loads of W_g), which also adds the partials and writes the gated
// representation g * m.  The CUDA-core bias kernel then reads that
// representation instead of gathering rows of E, and so does the verifier's
// residual pass.
//
// RNN head ("DSpark notes" 2.3, the second form; "DSpark 论文精读" 2.3,
// RNNHead): with u_j = [s_{j-1}; m_j; h_j],
//     g = sigmoid(W_g u), c = tanh(W_c u), s_j = g * s_{j-1} + (1 - g) * c,
//     o_j = tanh(W_o [s_j; m_j; h_j]),  b_j = W o_j,  s = 0 at the start.
// W_rnn is [3, rank, 2 rank + H] (W_g, W_c, W_o; columns: state, Markov
// row, hidden state).  The hidden-state parts of all three, for every
// position, are one dense product before the sequential stage (the same
// kernel as the gate's); each draft step then runs rnn_state_kernel (gate,
// candidate and state update: the state and Markov columns of W_g and W_c)
// and rnn_out_kernel (o_j from the new state), which writes the
// representation the bias kernel and the verifier's residual pass read.
#include "head_step.cuh"

namespace dsd {

namespace {

constexpr int kGhBM = 64, kGhBN = 64, kGhBK = 32, kGhThreads = 256;
constexpr int kGsOut = 8;          // outputs per CTA of the per-step kernels: one per warp

// Zh[s, n, k] = sum over c in split s (columns s width .. + width, below H)
// of h[n, c] Wh[k, c], for n < rows, k < n_out (width a multiple of 32),
// where row k of Wh starts at W + k ld + c_off.  The splits are summed in
// order by the step kernels, so the result does not depend on scheduling.
// H, ld and c_off are multiples of 8; a group of eight consecutive c is
// either wholly inside H or wholly outside.
template <typename T>
__global__ void __launch_bounds__(kGhThreads) gate_h_kernel(const T* __restrict__ h,
                                                            const T* __restrict__ W, int rows,
                                                            int H, int n_out, int ld, int c_off,
                                                            int width, float* Zh) {
  const int rank = n_out;   // output columns of Zh
  __shared__ __align__(16) float As[kGhBK][kGhBM + 4];
  __shared__ __align__(16) float Bs[kGhBK][kGhBN + 4];
  const int tid = threadIdx.x;
  const int n0 = blockIdx.y * kGhBM, k0 = blockIdx.x * kGhBN;
  const int tm = (tid / 16) * 4, tn = (tid % 16) * 4;   // this thread's 4 x 4 outputs
  float acc[4][4] = {};
  // loader: one group of 8 K-values of one row of A and of B per thread
  const int lr = tid / 4, lc = (tid % 4) * 8;
  const int cs = blockIdx.z * width, ce = min(H, cs + width);
  Zh += (size_t)blockIdx.z * rows * rank;
  for (int c0 = cs; c0 < ce; c0 += kGhBK) {
    float xa[8], xb[8];
    const int c = c0 + lc;
    const int na = n0 + lr, kb = k0 + lr;
    if (c < ce && na < rows) load8<T>(h + (size_t)na * H + c, xa);
    else for (int e = 0; e < 8; ++e) xa[e] = 0.f;
    if (c < ce && kb < rank) load8<T>(W + (size_t)kb * ld + c_off + c, xb);
    else for (int e = 0; e < 8; ++e) xb[e] = 0.f;
    __syncthreads();
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      As[lc + e][lr] = xa[e];
      Bs[lc + e][lr] = xb[e];
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kGhBK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[kk][tm]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tn]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = fmaf(av[i], bv[q], acc[i][q]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int n = n0 + tm + i;
    if (n >= rows) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int k = k0 + tn + q;
      if (k < rank) Zh[(size_t)n * rank + k] = acc[i][q];
    }
  }
}

// One CTA per request and 8 outputs, one warp per output.
template <typename T>
__global__ void __launch_bounds__(256) gate_step_kernel(HeadStepParams p, int j) {
  const int r = blockIdx.x, warp = threadIdx.x >> 5;
  const int k0 = blockIdx.y * kGsOut, k1 = min(p.rank, k0 + kGsOut);
  for (int k = k0 + warp; k < k1; k += blockDim.x / 32) gate_outputs_warp<T, 1>(p, j, r, k);
}

// Gate, candidate and state update of one step: CTA = one request and 8
// state units, one warp per unit.
template <typename T>
__global__ void __launch_bounds__(256) rnn_state_kernel(HeadStepParams p, int j) {
  const int r = blockIdx.x, warp = threadIdx.x >> 5;
  const int k0 = blockIdx.y * kGsOut, k1 = min(p.rank, k0 + kGsOut);
  for (int k = k0 + warp; k < k1; k += blockDim.x / 32) rnn_state_warp<T, 1>(p, j, r, k);
}

// Output of one step: o_j = tanh(W_o [s_j; m_j; h_j]), the representation
// the bias projection multiplies.
template <typename T>
__global__ void __launch_bounds__(256) rnn_out_kernel(HeadStepParams p, int j) {
  const int r = blockIdx.x, warp = threadIdx.x >> 5;
  const int k0 = blockIdx.y * kGsOut, k1 = min(p.rank, k0 + kGsOut);
  for (int k = k0 + warp; k < k1; k += blockDim.x / 32) rnn_out_warp<T, 1>(p, j, r, k);
}

}  // namespace

// Split of the hidden columns: enough CTAs to cover every SM, within the
// workspace (kGateZhFactor x R_max gamma x rank floats of partials) and at
// least 32 columns per split.
static void gate_split(const Ctx& ctx, int rows, int H, int n_out, int* n_split, int* width) {
  const int tiles = ((n_out + kGhBN - 1) / kGhBN) * ((rows + kGhBM - 1) / kGhBM);
  int n = (ctx.num_sms + tiles - 1) / tiles;
  const long long cap_floats = (long long)kGateZhFactor * ctx.cfg.R_max * ctx.cfg.gamma * ctx.cfg.rank;
  const long long per_split = (long long)(rows > 0 ? rows : 1) * n_out;
  const int cap = (int)(cap_floats / per_split);
  n = n < cap ? n : cap;
  const int most = (H + 31) / 32;
  n = n < most ? n : most;
  n = n < 1 ? 1 : n;
  int w = (H + n - 1) / n;
  w = (w + 31) / 32 * 32;
  *width = w;
  *n_split = (H + w - 1) / w;
}

// Hidden-state parts of every position: n_out weight rows of length H
// starting at column c_off of rows ld apart.
static cudaError_t launch_hidden(const Ctx& ctx, const ProposeArgs& a, const void* Wt, int n_out,
                                 int ld, int c_off, cudaStream_t s) {
  const int rows = a.R * a.gamma;
  int n_split, width;
  gate_split(ctx, rows, a.H, n_out, &n_split, &width);
  const dim3 grid((n_out + kGhBN - 1) / kGhBN, (rows + kGhBM - 1) / kGhBM, n_split);
  if (a.dtype == 1)
    gate_h_kernel<__nv_bfloat16><<<grid, kGhThreads, 0, s>>>(
        static_cast<const __nv_bfloat16*>(a.gate_h), static_cast<const __nv_bfloat16*>(Wt), rows,
        a.H, n_out, ld, c_off, width, ctx.ws.gate_zh);
  else
    gate_h_kernel<float><<<grid, kGhThreads, 0, s>>>(static_cast<const float*>(a.gate_h),
                                                     static_cast<const float*>(Wt), rows, a.H,
                                                     n_out, ld, c_off, width, ctx.ws.gate_zh);
  count_launch(ctx);
  return cudaGetLastError();
}

cudaError_t launch_gate_h(const Ctx& ctx, const ProposeArgs& a, cudaStream_t s) {
  return launch_hidden(ctx, a, a.W_g, a.rank, a.H + a.rank, 0, s);
}

HeadStepParams head_step_params(const Ctx& ctx, const ProposeArgs& a) {
  HeadStepParams p{};
  p.E = a.E;
  p.W = a.rnn_W ? a.rnn_W : a.W_g;
  p.Zh = ctx.ws.gate_zh;
  p.rows = a.R * a.gamma;
  int width;
  gate_split(ctx, p.rows, a.H, a.rnn_W ? 3 * a.rank : a.rank, &p.n_split, &width);
  p.prev_tok = a.prev_tok;
  p.keys = ctx.ws.keys;
  p.state = ctx.ws.rnn_state;
  p.A = a.gated_rep;
  p.status = ctx.ws.status;
  p.R_max = ctx.cfg.R_max;
  p.V = a.V;
  p.H = a.H;
  p.rank = a.rank;
  p.gamma = a.gamma;
  p.act = a.act;
  p.bias_at_first = a.bias_at_first;
  return p;
}

cudaError_t launch_gate_step(const Ctx& ctx, const ProposeArgs& a, int j, cudaStream_t s) {
  const HeadStepParams p = head_step_params(ctx, a);
  const dim3 grid(a.R, (a.rank + kGsOut - 1) / kGsOut);
  if (a.dtype == 1)
    gate_step_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(p, j);
  else
    gate_step_kernel<float><<<grid, 256, 0, s>>>(p, j);
  count_launch(ctx);
  return cudaGetLastError();
}

cudaError_t launch_rnn_h(const Ctx& ctx, const ProposeArgs& a, cudaStream_t s) {
  return launch_hidden(ctx, a, a.rnn_W, 3 * a.rank, 2 * a.rank + a.H, 2 * a.rank, s);
}

cudaError_t launch_rnn_step(const Ctx& ctx, const ProposeArgs& a, int j, cudaStream_t s) {
  const HeadStepParams p = head_step_params(ctx, a);
  const dim3 grid(a.R, (a.rank + kGsOut - 1) / kGsOut);
  if (a.dtype == 1) {
    rnn_state_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(p, j);
    rnn_out_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(p, j);
  } else {
    rnn_state_kernel<float><<<grid, 256, 0, s>>>(p, j);
    rnn_out_kernel<float><<<grid, 256, 0, s>>>(p, j);
  }
  count_launch(ctx, 2);
  return cudaGetLastError();
}

}  // namespace dsd
