// C-ABI entry points (include/dsd.h): context and workspace management,
// host-side argument validation, engine dispatch.  No compute happens here;
// every step of the path runs in the kernels of this directory.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <cmath>
#include <new>

#include <nvtx3/nvToolsExt.h>

#include "../../include/dsd.h"
#include "dsd_common.cuh"
#include "dsd_internal.h"

using namespace dsd;

struct dsd_ctx : public dsd::Ctx {};

namespace {

// One NVTX range per public call (named after the call), so a profiler's
// timeline shows which API call launched which kernels.  Without a tool
// attached a push or pop is a call through an empty hook.
struct Trace {
  explicit Trace(const char* name) { nvtxRangePushA(name); }
  ~Trace() { nvtxRangePop(); }
  Trace(const Trace&) = delete;
  Trace& operator=(const Trace&) = delete;
};

int fail(dsd_ctx* ctx, int code, const char* fmt, ...) {
  if (ctx) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(ctx->err, sizeof(ctx->err), fmt, ap);
    va_end(ap);
  }
  return code;
}

int cuda_fail(dsd_ctx* ctx, cudaError_t e, const char* where) {
  return fail(ctx, DSD_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Carve the workspace; with base == nullptr only computes the size.
size_t carve(dsd_ctx* c, unsigned char* base) {
  const int Rm = c->cfg.R_max, G = c->cfg.gamma;
  size_t off = 0;
  auto take = [&](size_t bytes) -> unsigned char* {
    unsigned char* p = base ? base + off : nullptr;
    off = align_up(off + bytes, 256);
    return p;
  };
  Workspace w{};
  w.status = reinterpret_cast<int*>(take(sizeof(int) * 4));
  w.counters = reinterpret_cast<unsigned int*>(take(sizeof(unsigned int) * 16));
  w.keys = reinterpret_cast<unsigned long long*>(
      take(sizeof(unsigned long long) * (size_t)G * Rm + sizeof(unsigned int) * kStepSyncWords));
  w.step_sync = w.keys ? reinterpret_cast<unsigned int*>(w.keys + (size_t)G * Rm) : nullptr;
  w.lse_parts = reinterpret_cast<float2*>(take(sizeof(float2) * (size_t)G * c->n_part * Rm));
  w.vparts = reinterpret_cast<RowPart*>(take(sizeof(RowPart) * (size_t)Rm * (G + 1) * kVerifySplits));
  w.rej_list = reinterpret_cast<int*>(take(sizeof(int) * (size_t)Rm));
  w.rej_k = reinterpret_cast<int*>(take(sizeof(int) * (size_t)Rm));
  w.rej_lseP = reinterpret_cast<float*>(take(sizeof(float) * (size_t)Rm));
  w.res_keys = reinterpret_cast<unsigned long long*>(take(sizeof(unsigned long long) * 2 * (size_t)Rm));
  w.res_sums = reinterpret_cast<float*>(take(sizeof(float) * 2 * (size_t)Rm));
  w.ov_parts = reinterpret_cast<float*>(take(sizeof(float) * 64));
  w.sched_theta = reinterpret_cast<unsigned long long*>(
      take(sizeof(unsigned long long) * (kMaxSchedItems + 1)));   // + the running maximum
  w.sched_order = reinterpret_cast<int*>(take(sizeof(int) * kMaxSchedItems));
  w.tickets = reinterpret_cast<unsigned int*>(take(sizeof(unsigned int) * 64));
  const size_t loss_rows = (size_t)Rm * G;
  w.loss_parts1 = reinterpret_cast<float4*>(take(sizeof(float4) * c->num_sms * loss_rows));
  w.loss_parts2 = reinterpret_cast<float*>(take(sizeof(float) * c->num_sms * loss_rows));
  w.loss_ltgt = reinterpret_cast<float*>(take(sizeof(float) * loss_rows));
  w.loss_red = reinterpret_cast<double*>(take(sizeof(double) * 64 * 3));
  w.cal_acc = reinterpret_cast<double*>(take(sizeof(double) * (2 * kMaxCalBins + 2 + 2 * kMaxGamma)));
  w.cal_cnt = reinterpret_cast<unsigned long long*>(take(sizeof(unsigned long long) * (kMaxCalBins + 1)));
  // split-K partials of the gate's hidden-state part
  w.gate_zh = reinterpret_cast<float*>(take(sizeof(float) * kGateZhFactor * (size_t)Rm * G * c->cfg.rank));
  w.rnn_state = reinterpret_cast<float*>(take(sizeof(float) * 2 * (size_t)Rm * c->cfg.rank));
  const int cand_R = Rm < kCandMaxR ? Rm : kCandMaxR;
  w.cand_parts = reinterpret_cast<unsigned long long*>(
      take(sizeof(unsigned long long) * (size_t)G * c->n_part * cand_R * kCandK));
  if (base) c->ws = w;
  return off;
}

int check_ctx(dsd_ctx* ctx) {
  if (!ctx) return DSD_ERR_ARG;
  ctx->err[0] = 0;
  cudaError_t e = cudaSetDevice(ctx->cfg.device);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaSetDevice");
  return DSD_OK;
}

int check_table(dsd_ctx* ctx, const void* p, const char* name) {
  if (!p) return fail(ctx, DSD_ERR_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(ctx, DSD_ERR_ALIGN, "%s is not 16-byte aligned", name);
  return DSD_OK;
}

int check_R(dsd_ctx* ctx, int R) {
  if (R < 0) return fail(ctx, DSD_ERR_ARG, "R = %d < 0", R);
  if (R > ctx->cfg.R_max) return fail(ctx, DSD_ERR_SHAPE, "R = %d > R_max = %d", R, ctx->cfg.R_max);
  return DSD_OK;
}

int check_temperature(dsd_ctx* ctx, float T) {
  if (!(T >= 0.f) || T != T || T > 3.0e38f)
    return fail(ctx, DSD_ERR_ARG, "temperature must be finite and >= 0");
  return DSD_OK;
}

// The warp-level tensor-core engine needs bf16 operands with no activation
// (the gathered rows are used as stored) and a rank that is a multiple of 64.
bool mma_ok(const dsd_ctx* ctx) {
  return ctx->cfg.dtype == DSD_BF16 && ctx->cfg.rank % 64 == 0 && ctx->cfg.rank <= 256 &&
         ctx->cfg.act == DSD_ACT_NONE;
}

}  // namespace

namespace dsd {
int simt_grid(const Ctx& ctx, int V);
cudaError_t launch_propose_finalize_n(const Ctx& ctx, const ProposeArgs& a, int n_used,
                                      cudaStream_t s);
int tc_supported(const Ctx& ctx, char* why, size_t why_len);
int tc_vranges(const Ctx& ctx, int R);
int tc_parts_used(const Ctx& ctx, const ProposeArgs& a);
}  // namespace dsd

namespace {
// AUTO sends every batch to the tcgen05 engine when the configuration
// allows it (bf16 tables, rank a multiple of 64 <= 256; an activation runs in
// its split mode): even one request drafts about 3x faster there than on the
// CUDA-core engine, whose per-tile shared-memory traffic does not shrink
// with R.
bool auto_uses_tc(const dsd_ctx* ctx, int R) {
  if (ctx->cfg.engine != DSD_ENGINE_AUTO || R < 1) return false;
  char why[256];
  return dsd::tc_supported(*ctx, why, sizeof(why)) != 0;
}
}  // namespace

extern "C" {

int dsd_create(const dsd_config* cfg, dsd_ctx** out) {
  if (!cfg || !out) return DSD_ERR_ARG;
  if (cfg->V < 8 || cfg->V % 8 != 0) return DSD_ERR_ALIGN;
  const bool rank_ok = (cfg->rank % 64 == 0 && cfg->rank <= 256) ||
                       (cfg->rank > 0 && cfg->rank <= 64 && cfg->rank % 8 == 0);
  if (!rank_ok) return DSD_ERR_SHAPE;
  if (cfg->gamma < 1 || cfg->gamma > kMaxGamma) return DSD_ERR_SHAPE;
  if (cfg->R_max < 1 || (long long)cfg->R_max * cfg->gamma > kMaxSchedItems) return DSD_ERR_SHAPE;
  if (cfg->dtype != DSD_F32 && cfg->dtype != DSD_BF16) return DSD_ERR_DTYPE;
  if (cfg->act != DSD_ACT_NONE && cfg->act != DSD_ACT_SILU) return DSD_ERR_ARG;
  if (cfg->engine < DSD_ENGINE_AUTO || cfg->engine > DSD_ENGINE_MMA) return DSD_ERR_ARG;
  if ((cfg->engine == DSD_ENGINE_TCGEN05 || cfg->engine == DSD_ENGINE_MMA) &&
      cfg->dtype != DSD_BF16)
    return DSD_ERR_DTYPE;

  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || cfg->device < 0 || cfg->device >= ndev)
    return DSD_ERR_UNSUPPORTED;
  if (cudaSetDevice(cfg->device) != cudaSuccess) return DSD_ERR_CUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, cfg->device) != cudaSuccess) return DSD_ERR_CUDA;
  if (prop.major != 10) return DSD_ERR_UNSUPPORTED;

  dsd_ctx* c = new (std::nothrow) dsd_ctx();
  if (!c) return DSD_ERR_ARG;
  memset(static_cast<dsd::Ctx*>(c), 0, sizeof(dsd::Ctx));
  c->cfg = Config{cfg->V, cfg->rank, cfg->gamma, cfg->R_max, cfg->dtype,
                  cfg->act, cfg->bias_at_first ? 1 : 0, cfg->engine, cfg->device};
  c->num_sms = prop.multiProcessorCount;
  c->n_part = 2 * c->num_sms;
  const size_t bytes = carve(c, nullptr);
  void* base = nullptr;
  if (cudaMalloc(&base, bytes) != cudaSuccess) {
    delete c;
    return DSD_ERR_CUDA;
  }
  if (cudaMemset(base, 0, bytes) != cudaSuccess) {
    cudaFree(base);
    delete c;
    return DSD_ERR_CUDA;
  }
  c->ws_base = base;
  c->ws_bytes = bytes;
  carve(c, static_cast<unsigned char*>(base));
  *out = c;
  return DSD_OK;
}

int dsd_destroy(dsd_ctx* ctx) {
  if (!ctx) return DSD_OK;
  cudaSetDevice(ctx->cfg.device);
  if (ctx->ws_base) cudaFree(ctx->ws_base);
  if (ctx->stage_base) cudaFree(ctx->stage_base);
  delete ctx;
  return DSD_OK;
}

const char* dsd_last_error(const dsd_ctx* ctx) { return ctx ? ctx->err : "null context"; }

size_t dsd_workspace_bytes(const dsd_ctx* ctx) { return ctx ? ctx->ws_bytes : 0; }

uint64_t dsd_launch_count(const dsd_ctx* ctx) { return ctx ? ctx->launches : 0; }

int dsd_last_engine(const dsd_ctx* ctx) { return ctx ? ctx->last_engine : 0; }
int dsd_last_p_in_place(const dsd_ctx* ctx) { return ctx ? ctx->last_p_in_place : 0; }

static __global__ void gumbel_noise_kernel(const uint32_t* words, float* out, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    out[i] = dsd::gumbel_from_word(words[i]);
}

int dsd_gumbel_noise(const uint32_t* words, float* out, int n, void* stream) {
  Trace trace_("dsd_gumbel_noise");
  if (n < 0 || (n > 0 && (!words || !out))) return DSD_ERR_ARG;
  if (n == 0) return DSD_OK;
  const int grid = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
  gumbel_noise_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(words, out, n);
  return cudaGetLastError() == cudaSuccess ? DSD_OK : DSD_ERR_CUDA;
}

int dsd_wait_selftest(dsd_ctx* ctx, uint32_t poll_limit, int32_t* roles_out, void* stream) {
  Trace trace_("dsd_wait_selftest");
  int rc = check_ctx(ctx);
  if (rc) return rc;
  if (poll_limit == 0 || poll_limit > (1u << 20))
    return fail(ctx, DSD_ERR_ARG, "poll_limit %u outside [1, 2^20]", poll_limit);
  cudaError_t e = dsd::launch_wait_selftest(*ctx, poll_limit, roles_out,
                                            static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(ctx, e, "wait self-test launch");
  return DSD_OK;
}

int dsd_sync_status(dsd_ctx* ctx, void* stream) {
  Trace trace_("dsd_sync_status");
  int rc = check_ctx(ctx);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaStreamSynchronize");
  int st = 0;
  e = cudaMemcpy(&st, ctx->ws.status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "read status");
  if (st != 0) {
    e = cudaMemset(ctx->ws.status, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(ctx, e, "clear status");
    fail(ctx, st, "device reported status %d", st);
  }
  return st;
}

// dsd_propose, optionally with the cycle's schedule folded into the
// finalize launch (sps != nullptr).
static int propose_impl(dsd_ctx* ctx, int R, const void* U, const void* E, const void* W,
                        const float* conf, const int32_t* prev_tok, const uint32_t* req_id,
                        float temperature, uint64_t seed, int32_t* tokens, float* lse_q,
                        float* logit_at_tok, float* survival, const float* sps, int n_sps,
                        int32_t* keep_len, float* theta_B, void* stream) {
  int rc = check_ctx(ctx);
  if (rc) return rc;
  if ((rc = check_R(ctx, R))) return rc;
  if ((rc = check_temperature(ctx, temperature))) return rc;
  if (R == 0) return DSD_OK;
  if ((rc = check_table(ctx, U, "U")) || (rc = check_table(ctx, E, "E")) ||
      (rc = check_table(ctx, W, "W")))
    return rc;
  if (!conf || !prev_tok || !tokens || !lse_q || !logit_at_tok || !survival)
    return fail(ctx, DSD_ERR_ARG, "dsd_propose: NULL argument");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ProposeArgs a{};
  a.R = R;
  a.V = ctx->cfg.V;
  a.rank = ctx->cfg.rank;
  a.gamma = ctx->cfg.gamma;
  a.dtype = ctx->cfg.dtype;
  a.act = ctx->cfg.act;
  a.bias_at_first = ctx->cfg.bias_at_first;
  a.U = U;
  a.E = E;
  a.W = W;
  a.conf = conf;
  a.prev_tok = prev_tok;
  a.req_id = req_id;
  a.temperature = temperature;
  a.seed = seed;
  a.tokens = tokens;
  a.lse_q = lse_q;
  a.logit_at_tok = logit_at_tok;
  a.survival = survival;
  if (sps) {
    a.sched_sps = sps;
    a.sched_n_sps = n_sps;
    a.sched_keep = keep_len;
    a.sched_theta = theta_B;
  }
  cudaError_t e;
  int n_used;
  if (ctx->cfg.engine == DSD_ENGINE_TCGEN05 || auto_uses_tc(ctx, R)) {
    char why[256];
    if (!tc_supported(*ctx, why, sizeof(why))) return fail(ctx, DSD_ERR_UNSUPPORTED, "%s", why);
    e = launch_propose_tc(*ctx, a, s);
    n_used = tc_parts_used(*ctx, a);
    ctx->last_engine = DSD_ENGINE_TCGEN05;
  } else if (ctx->cfg.engine == DSD_ENGINE_MMA && !mma_ok(ctx)) {
    return fail(ctx, DSD_ERR_UNSUPPORTED,
                "MMA engine needs bf16 tables, no activation and rank %% 64 == 0 (<= 256)");
  } else if (ctx->cfg.engine == DSD_ENGINE_MMA) {
    e = launch_propose_mma(*ctx, a, s);
    n_used = mma_vranges(*ctx, R);
    ctx->last_engine = DSD_ENGINE_MMA;
  } else {
    e = launch_propose_simt(*ctx, a, s);
    n_used = simt_grid(*ctx, a.V);
    ctx->last_engine = DSD_ENGINE_SIMT;
  }
  if (e != cudaSuccess) return cuda_fail(ctx, e, "propose launch");
  e = launch_propose_finalize_n(*ctx, a, n_used, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "propose finalize launch");
  return DSD_OK;
}

int dsd_propose(dsd_ctx* ctx, int R, const void* U, const void* E, const void* W,
                const float* conf, const int32_t* prev_tok, const uint32_t* req_id,
                float temperature, uint64_t seed, int32_t* tokens, float* lse_q,
                float* logit_at_tok, float* survival, void* stream) {
  Trace trace_("dsd_propose");
  return propose_impl(ctx, R, U, E, W, conf, prev_tok, req_id, temperature, seed, tokens, lse_q,
                      logit_at_tok, survival, nullptr, 0, nullptr, nullptr, stream);
}

int dsd_schedule(dsd_ctx* ctx, int R, const float* survival, const float* sps, int n_sps,
                 int32_t* keep_len, float* theta_B, void* stream) {
  Trace trace_("dsd_schedule");
  int rc = check_ctx(ctx);
  if (rc) return rc;
  if ((rc = check_R(ctx, R))) return rc;
  if (R == 0) return DSD_OK;
  if (!survival || !sps || !keep_len) return fail(ctx, DSD_ERR_ARG, "dsd_schedule: NULL argument");
  if (n_sps < 1) return fail(ctx, DSD_ERR_ARG, "n_sps = %d", n_sps);
  if (R > n_sps) return fail(ctx, DSD_ERR_CAPACITY, "R = %d exceeds the SPS table (%d)", R, n_sps);
  cudaError_t e = launch_schedule(*ctx, R, survival, sps, n_sps, keep_len, theta_B,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(ctx, e, "schedule launch");
  return DSD_OK;
}

static int verify_impl(dsd_ctx* ctx, int R, const void* P, const void* U, const void* E,
                       const void* W, const int32_t* prev_tok, const int32_t* tokens,
                       const float* lse_q, const float* logit_at_tok, const int32_t* keep_len,
                       const uint32_t* req_id, float temperature, uint64_t seed,
                       int32_t* accept_len, int32_t* next_token, const float* gated_rep,
                       void* stream) {
  int rc = check_ctx(ctx);
  if (rc) return rc;
  if ((rc = check_R(ctx, R))) return rc;
  if ((rc = check_temperature(ctx, temperature))) return rc;
  if (R == 0) return DSD_OK;
  if ((rc = check_table(ctx, P, "P"))) return rc;
  if (!tokens || !keep_len || !accept_len || !next_token)
    return fail(ctx, DSD_ERR_ARG, "dsd_verify: NULL argument");
  if (temperature > 0.f) {
    if ((rc = check_table(ctx, U, "U")) || (rc = check_table(ctx, E, "E")) ||
        (rc = check_table(ctx, W, "W")))
      return rc;
    if (!prev_tok || !lse_q || !logit_at_tok)
      return fail(ctx, DSD_ERR_ARG, "dsd_verify: sampled mode needs prev_tok, lse_q, logit_at_tok");
  }
  VerifyArgs a{};
  a.R = R;
  a.V = ctx->cfg.V;
  a.rank = ctx->cfg.rank;
  a.gamma = ctx->cfg.gamma;
  a.dtype = ctx->cfg.dtype;
  a.act = ctx->cfg.act;
  a.bias_at_first = ctx->cfg.bias_at_first;
  a.P = P;
  a.U = U;
  a.E = E;
  a.W = W;
  a.prev_tok = prev_tok;
  a.tokens = tokens;
  a.lse_q = lse_q;
  a.logit_at_tok = logit_at_tok;
  a.keep_len = keep_len;
  a.req_id = req_id;
  a.temperature = temperature;
  a.seed = seed;
  a.accept_len = accept_len;
  a.next_token = next_token;
  a.gated_rep = gated_rep;
  cudaError_t e = launch_verify(*ctx, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(ctx, e, "verify launch");
  return DSD_OK;
}

int dsd_verify(dsd_ctx* ctx, int R, const void* P, const void* U, const void* E, const void* W,
               const int32_t* prev_tok, const int32_t* tokens, const float* lse_q,
               const float* logit_at_tok, const int32_t* keep_len, const uint32_t* req_id,
               float temperature, uint64_t seed, int32_t* accept_len, int32_t* next_token,
               void* stream) {
  Trace trace_("dsd_verify");
  return verify_impl(ctx, R, P, U, E, W, prev_tok, tokens, lse_q, logit_at_tok, keep_len, req_id,
                     temperature, seed, accept_len, next_token, nullptr, stream);
}

int dsd_verify_rnn(dsd_ctx* ctx, int R, const void* P, const void* U, const void* E,
                   const void* W, const float* rnn_rep, const int32_t* prev_tok,
                   const int32_t* tokens, const float* lse_q, const float* logit_at_tok,
                   const int32_t* keep_len, const uint32_t* req_id, float temperature,
                   uint64_t seed, int32_t* accept_len, int32_t* next_token, void* stream) {
  Trace trace_("dsd_verify_rnn");
  int rc = check_ctx(ctx);
  if (rc) return rc;
  if (R > 0 && temperature > 0.f && !rnn_rep)
    return fail(ctx, DSD_ERR_ARG, "dsd_verify_rnn: rnn_rep is NULL");
  return verify_impl(ctx, R, P, U, E, W, prev_tok, tokens, lse_q, logit_at_tok, keep_len, req_id,
                     temperature, seed, accept_len, next_token, rnn_rep, stream);
}

int dsd_verify_gated(dsd_ctx* ctx, int R, const void* P, const void* U, const void* E,
                     const void* W, const float* gated_rep, const int32_t* prev_tok,
                     const int32_t* tokens, const float* lse_q, const float* logit_at_tok,
                     const int32_t* keep_len, const uint32_t* req_id, float temperature,
                     uint64_t seed, int32_t* accept_len, int32_t* next_token, void* stream) {
  Trace trace_("dsd_verify_gated");
  int rc = check_ctx(ctx);
  if (rc) return rc;
  if (R > 0 && temperature > 0.f && !gated_rep)
    return fail(ctx, DSD_ERR_ARG, "dsd_verify_gated: gated_rep is NULL");
  return verify_impl(ctx, R, P, U, E, W, prev_tok, tokens, lse_q, logit_at_tok, keep_len, req_id,
                     temperature, seed, accept_len, next_token, gated_rep, stream);
}

// The heads that read the backbone's hidden state: the gated Markov head
// (W_g) or the RNN head (W_rnn).  Their per-step representation is fp32, so
// the tensor-core engine runs them in its split mode (hi and lo bf16 parts);
// the SIMT engine, or a configuration it cannot take, uses the CUDA cores.
static int propose_hidden_head(dsd_ctx* ctx, const char* name, int R, const void* U,
                               const void* E, const void* W, const void* h, int H,
                               const void* W_g, const void* W_rnn, const float* conf,
                               const int32_t* prev_tok, const uint32_t* req_id,
                               float temperature, uint64_t seed, int32_t* tokens, float* lse_q,
                               float* logit_at_tok, float* survival, float* rep, void* stream) {
  int rc = check_ctx(ctx);
  if (rc) return rc;
  if ((rc = check_R(ctx, R))) return rc;
  if ((rc = check_temperature(ctx, temperature))) return rc;
  if (H <= 0 || H % 8 != 0) return fail(ctx, DSD_ERR_ALIGN, "H = %d must be a positive multiple of 8", H);
  if (R == 0) return DSD_OK;
  if ((rc = check_table(ctx, U, "U")) || (rc = check_table(ctx, E, "E")) ||
      (rc = check_table(ctx, W, "W")) || (rc = check_table(ctx, h, "h")) ||
      (rc = check_table(ctx, W_g ? W_g : W_rnn, W_g ? "W_g" : "W_rnn")))
    return rc;
  if (!conf || !prev_tok || !tokens || !lse_q || !logit_at_tok || !survival || !rep)
    return fail(ctx, DSD_ERR_ARG, "%s: NULL argument", name);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ProposeArgs a{};
  a.R = R;
  a.V = ctx->cfg.V;
  a.rank = ctx->cfg.rank;
  a.gamma = ctx->cfg.gamma;
  a.dtype = ctx->cfg.dtype;
  a.act = ctx->cfg.act;
  a.bias_at_first = ctx->cfg.bias_at_first;
  a.U = U;
  a.E = E;
  a.W = W;
  a.conf = conf;
  a.prev_tok = prev_tok;
  a.req_id = req_id;
  a.temperature = temperature;
  a.seed = seed;
  a.tokens = tokens;
  a.lse_q = lse_q;
  a.logit_at_tok = logit_at_tok;
  a.survival = survival;
  a.gate_h = h;
  a.W_g = W_g;
  a.rnn_W = W_rnn;
  a.H = H;
  a.gated_rep = rep;
  char why[256];
  const bool tc = (ctx->cfg.engine == DSD_ENGINE_AUTO || ctx->cfg.engine == DSD_ENGINE_TCGEN05) &&
                  tc_supported(*ctx, why, sizeof(why));
  if (ctx->cfg.engine == DSD_ENGINE_TCGEN05 && !tc)
    return fail(ctx, DSD_ERR_UNSUPPORTED, "%s", why);
  cudaError_t e = tc ? launch_propose_tc(*ctx, a, s) : launch_propose_simt(*ctx, a, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, name);
  ctx->last_engine = tc ? DSD_ENGINE_TCGEN05 : DSD_ENGINE_SIMT;
  e = launch_propose_finalize_n(*ctx, a, tc ? tc_parts_used(*ctx, a) : simt_grid(*ctx, a.V), s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "propose finalize launch");
  return DSD_OK;
}

int dsd_propose_gated(dsd_ctx* ctx, int R, const void* U, const void* E, const void* W,
                      const void* h, int H, const void* W_g, const float* conf,
                      const int32_t* prev_tok, const uint32_t* req_id, float temperature,
                      uint64_t seed, int32_t* tokens, float* lse_q, float* logit_at_tok,
                      float* survival, float* gated_rep, void* stream) {
  Trace trace_("dsd_propose_gated");
  if (ctx && !W_g) return fail(ctx, DSD_ERR_ARG, "dsd_propose_gated: W_g is NULL");
  return propose_hidden_head(ctx, "dsd_propose_gated", R, U, E, W, h, H, W_g, nullptr, conf,
                             prev_tok, req_id, temperature, seed, tokens, lse_q, logit_at_tok,
                             survival, gated_rep, stream);
}

int dsd_propose_rnn(dsd_ctx* ctx, int R, const void* U, const void* E, const void* W,
                    const void* h, int H, const void* W_rnn, const float* conf,
                    const int32_t* prev_tok, const uint32_t* req_id, float temperature,
                    uint64_t seed, int32_t* tokens, float* lse_q, float* logit_at_tok,
                    float* survival, float* rnn_rep, void* stream) {
  Trace trace_("dsd_propose_rnn");
  if (ctx && !W_rnn) return fail(ctx, DSD_ERR_ARG, "dsd_propose_rnn: W_rnn is NULL");
  return propose_hidden_head(ctx, "dsd_propose_rnn", R, U, E, W, h, H, nullptr, W_rnn, conf,
                             prev_tok, req_id, temperature, seed, tokens, lse_q, logit_at_tok,
                             survival, rnn_rep, stream);
}

int dsd_cycle(dsd_ctx* ctx, int R, const void* U, const void* E, const void* W, const float* conf,
              const int32_t* prev_tok, const uint32_t* req_id, const void* P, const float* sps,
              int n_sps, float temperature, uint64_t seed, int32_t* tokens, float* lse_q,
              float* logit_at_tok, float* survival, int32_t* keep_len, float* theta_B,
              int32_t* accept_len, int32_t* next_token, void* stream) {
  Trace trace_("dsd_cycle");
  // the schedule depends on the confidences only: it runs in extra CTAs of
  // the proposal's finalize launch
  int rc = check_ctx(ctx);
  if (rc) return rc;
  if ((rc = check_R(ctx, R))) return rc;
  if (R == 0) return DSD_OK;
  if (!sps || !keep_len) return fail(ctx, DSD_ERR_ARG, "dsd_cycle: NULL argument");
  if (n_sps < 1) return fail(ctx, DSD_ERR_ARG, "n_sps = %d", n_sps);
  if (R > n_sps) return fail(ctx, DSD_ERR_CAPACITY, "R = %d exceeds the SPS table (%d)", R, n_sps);
  // verification's own argument checks, before the proposal launches
  // anything (the proposal's checks cover U, E, W, conf and prev_tok)
  if ((rc = check_table(ctx, P, "P"))) return rc;
  if (!accept_len || !next_token) return fail(ctx, DSD_ERR_ARG, "dsd_cycle: NULL argument");
  rc = propose_impl(ctx, R, U, E, W, conf, prev_tok, req_id, temperature, seed, tokens, lse_q,
                    logit_at_tok, survival, sps, n_sps, keep_len, theta_B, stream);
  if (rc) return rc;
  return dsd_verify(ctx, R, P, U, E, W, prev_tok, tokens, lse_q, logit_at_tok, keep_len, req_id,
                    temperature, seed, accept_len, next_token, stream);
}

int dsd_cycle_host(dsd_ctx* ctx, int R, const void* U_host, const void* E, const void* W,
                   const float* conf_host, const int32_t* prev_tok_host,
                   const uint32_t* req_id_host, const void* P_host, const float* sps, int n_sps,
                   float temperature, uint64_t seed, int32_t* tokens_host, int32_t* keep_len_host,
                   int32_t* accept_len_host, int32_t* next_token_host, void* stream) {
  Trace trace_("dsd_cycle_host");
  int rc = check_ctx(ctx);
  if (rc) return rc;
  if ((rc = check_R(ctx, R))) return rc;
  if (R == 0) return DSD_OK;
  if (!U_host || !conf_host || !prev_tok_host || !P_host || !tokens_host || !keep_len_host ||
      !accept_len_host || !next_token_host)
    return fail(ctx, DSD_ERR_ARG, "dsd_cycle_host: NULL argument");
  const int Rm = ctx->cfg.R_max, G = ctx->cfg.gamma;
  const size_t V = (size_t)ctx->cfg.V;
  const size_t esz = ctx->cfg.dtype == DSD_BF16 ? 2 : 4;
  // staging layout: U, P, conf, prev, req, tokens, lse, logit, surv, keep, theta, acc, next
  size_t off = 0;
  size_t o_U = off; off = align_up(off + (size_t)Rm * G * V * esz, 256);
  size_t o_P = off; off = align_up(off + (size_t)Rm * (G + 1) * V * esz, 256);
  size_t o_conf = off; off = align_up(off + sizeof(float) * Rm * G, 256);
  size_t o_prev = off; off = align_up(off + sizeof(int32_t) * Rm, 256);
  size_t o_req = off; off = align_up(off + sizeof(uint32_t) * Rm, 256);
  size_t o_tok = off; off = align_up(off + sizeof(int32_t) * Rm * G, 256);
  size_t o_lse = off; off = align_up(off + sizeof(float) * Rm * G, 256);
  size_t o_lg = off; off = align_up(off + sizeof(float) * Rm * G, 256);
  size_t o_sv = off; off = align_up(off + sizeof(float) * Rm * G, 256);
  size_t o_keep = off; off = align_up(off + sizeof(int32_t) * Rm, 256);
  size_t o_th = off; off = align_up(off + sizeof(float) * 2, 256);
  size_t o_acc = off; off = align_up(off + sizeof(int32_t) * Rm, 256);
  size_t o_nx = off; off = align_up(off + sizeof(int32_t) * Rm, 256);
  if (!ctx->stage_base) {
    cudaError_t e = cudaMalloc(&ctx->stage_base, off);
    if (e != cudaSuccess) {
      ctx->stage_base = nullptr;
      return cuda_fail(ctx, e, "staging cudaMalloc");
    }
    ctx->stage_bytes = off;
  }
  unsigned char* b = static_cast<unsigned char*>(ctx->stage_base);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  const size_t G1 = (size_t)G + 1;
#define DSD_CPY(dst, src, bytes, kind)                                   \
  do {                                                                   \
    e = cudaMemcpyAsync((dst), (src), (bytes), (kind), s);               \
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaMemcpyAsync");   \
  } while (0)
  DSD_CPY(b + o_U, U_host, (size_t)R * G * V * esz, cudaMemcpyHostToDevice);
  // P is read in place when the GPU can address the caller's (pinned) host
  // buffer: verification reads only the kept rows, so only those cross the
  // CPU-GPU link.  Otherwise (pageable memory) the whole of P is staged.
  const void* P_dev = nullptr;
  {
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, P_host) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
        pa.devicePointer != nullptr && aligned16(pa.devicePointer))
      P_dev = pa.devicePointer;
    else
      (void)cudaGetLastError();
  }
  if (!P_dev) {
    DSD_CPY(b + o_P, P_host, (size_t)R * G1 * V * esz, cudaMemcpyHostToDevice);
    P_dev = b + o_P;
  }
  ctx->last_p_in_place = (P_dev != b + o_P) ? 1 : 0;
  DSD_CPY(b + o_conf, conf_host, sizeof(float) * R * G, cudaMemcpyHostToDevice);
  DSD_CPY(b + o_prev, prev_tok_host, sizeof(int32_t) * R, cudaMemcpyHostToDevice);
  if (req_id_host) DSD_CPY(b + o_req, req_id_host, sizeof(uint32_t) * R, cudaMemcpyHostToDevice);
  rc = dsd_cycle(ctx, R, b + o_U, E, W, reinterpret_cast<float*>(b + o_conf),
                 reinterpret_cast<int32_t*>(b + o_prev),
                 req_id_host ? reinterpret_cast<uint32_t*>(b + o_req) : nullptr, P_dev, sps,
                 n_sps, temperature, seed, reinterpret_cast<int32_t*>(b + o_tok),
                 reinterpret_cast<float*>(b + o_lse), reinterpret_cast<float*>(b + o_lg),
                 reinterpret_cast<float*>(b + o_sv), reinterpret_cast<int32_t*>(b + o_keep),
                 reinterpret_cast<float*>(b + o_th), reinterpret_cast<int32_t*>(b + o_acc),
                 reinterpret_cast<int32_t*>(b + o_nx), stream);
  if (rc) return rc;
  DSD_CPY(tokens_host, b + o_tok, sizeof(int32_t) * R * G, cudaMemcpyDeviceToHost);
  DSD_CPY(keep_len_host, b + o_keep, sizeof(int32_t) * R, cudaMemcpyDeviceToHost);
  DSD_CPY(accept_len_host, b + o_acc, sizeof(int32_t) * R, cudaMemcpyDeviceToHost);
  DSD_CPY(next_token_host, b + o_nx, sizeof(int32_t) * R, cudaMemcpyDeviceToHost);
#undef DSD_CPY
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaStreamSynchronize");
  return DSD_OK;
}

int dsd_overlap(dsd_ctx* ctx, int N, const void* P_logits, const void* Q_logits,
                const int32_t* valid_len, float* a, float* l1, float* tau, float* accept_rate,
                float* mean_tau, void* stream) {
  Trace trace_("dsd_overlap");
  int rc = check_ctx(ctx);
  if (rc) return rc;
  if (N < 0) return fail(ctx, DSD_ERR_ARG, "N = %d < 0", N);
  if (!accept_rate || !mean_tau) return fail(ctx, DSD_ERR_ARG, "dsd_overlap: NULL argument");
  if (N > 0) {
    if ((rc = check_table(ctx, P_logits, "P_logits")) || (rc = check_table(ctx, Q_logits, "Q_logits")))
      return rc;
    if (!valid_len || !a || !l1 || !tau) return fail(ctx, DSD_ERR_ARG, "dsd_overlap: NULL argument");
    if ((long long)N * ctx->cfg.gamma > 0x7fffffffLL) return fail(ctx, DSD_ERR_SHAPE, "N too large");
  }
  OverlapArgs o{};
  o.N = N;
  o.V = ctx->cfg.V;
  o.gamma = ctx->cfg.gamma;
  o.dtype = ctx->cfg.dtype;
  o.P = P_logits;
  o.Q = Q_logits;
  o.valid_len = valid_len;
  o.a = a;
  o.l1 = l1;
  o.tau = tau;
  o.accept_rate = accept_rate;
  o.mean_tau = mean_tau;
  cudaError_t e = launch_overlap(*ctx, o, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(ctx, e, "overlap launch");
  return DSD_OK;
}

int dsd_loss_forward(dsd_ctx* ctx, int B, const void* U, const void* E, const void* W,
                     const int32_t* prev_tok, const void* P, const int32_t* target,
                     const float* conf_logit, float ce_alpha, float l1_alpha, float conf_alpha,
                     float decay, float* row_out, float* losses, void* stream) {
  Trace trace_("dsd_loss_forward");
  int rc = check_ctx(ctx);
  if (rc) return rc;
  if ((rc = check_R(ctx, B))) return rc;
  if (!losses) return fail(ctx, DSD_ERR_ARG, "dsd_loss_forward: losses is NULL");
  const float fs[3] = {ce_alpha, l1_alpha, conf_alpha};
  for (float f : fs)
    if (!(f == f) || f > 3.0e38f || f < -3.0e38f)
      return fail(ctx, DSD_ERR_ARG, "dsd_loss_forward: loss weights must be finite");
  if (!(decay > 0.f) || decay > 3.0e38f)
    return fail(ctx, DSD_ERR_ARG, "dsd_loss_forward: decay must be finite and > 0");
  char why[256];
  if (!dsd::tc_supported(*ctx, why, sizeof(why)))
    return fail(ctx, DSD_ERR_UNSUPPORTED, "dsd_loss_forward: %s", why);
  if (ctx->cfg.act != DSD_ACT_NONE)   // its A operand is the stored bf16 rows of E
    return fail(ctx, DSD_ERR_UNSUPPORTED, "dsd_loss_forward runs without an activation");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (B == 0) {
    cudaError_t e = cudaMemsetAsync(losses, 0, 4 * sizeof(float), s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "loss memset");
    return DSD_OK;
  }
  if ((rc = check_table(ctx, U, "U")) || (rc = check_table(ctx, E, "E")) ||
      (rc = check_table(ctx, W, "W")) || (rc = check_table(ctx, P, "P")))
    return rc;
  if (!prev_tok || !target || !conf_logit)
    return fail(ctx, DSD_ERR_ARG, "dsd_loss_forward: NULL argument");
  LossArgs a{};
  a.B = B;
  a.V = ctx->cfg.V;
  a.rank = ctx->cfg.rank;
  a.gamma = ctx->cfg.gamma;
  a.bias_at_first = ctx->cfg.bias_at_first;
  a.U = U;
  a.E = E;
  a.W = W;
  a.P = P;
  a.prev_tok = prev_tok;
  a.target = target;
  a.conf_logit = conf_logit;
  a.ce_alpha = ce_alpha;
  a.l1_alpha = l1_alpha;
  a.conf_alpha = conf_alpha;
  a.decay = decay;
  a.row_out = row_out;
  a.losses = losses;
  cudaError_t e = launch_loss(*ctx, a, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "loss launch");
  return DSD_OK;
}

int dsd_confidence_head(dsd_ctx* ctx, int R, int H, const void* h, const void* E, const void* w_c,
                        float b_c, const int32_t* prev_tok, const int32_t* tokens, float* conf,
                        float* survival, void* stream) {
  Trace trace_("dsd_confidence_head");
  int rc = check_ctx(ctx);
  if (rc) return rc;
  if (R < 0) return fail(ctx, DSD_ERR_ARG, "R = %d < 0", R);
  if (H <= 0 || H % 8 != 0) return fail(ctx, DSD_ERR_ALIGN, "H = %d must be a positive multiple of 8", H);
  if (!std::isfinite(b_c)) return fail(ctx, DSD_ERR_NONFINITE, "b_c is not finite");
  if (R == 0) return DSD_OK;
  if ((long long)R * ctx->cfg.gamma > 0x7fffffffLL) return fail(ctx, DSD_ERR_SHAPE, "R too large");
  if ((rc = check_table(ctx, h, "h")) || (rc = check_table(ctx, E, "E")) ||
      (rc = check_table(ctx, w_c, "w_c")))
    return rc;
  if (!prev_tok || !tokens || !conf || !survival)
    return fail(ctx, DSD_ERR_ARG, "dsd_confidence_head: NULL argument");
  ConfHeadArgs a{};
  a.R = R;
  a.H = H;
  a.V = ctx->cfg.V;
  a.rank = ctx->cfg.rank;
  a.gamma = ctx->cfg.gamma;
  a.dtype = ctx->cfg.dtype;
  a.h = h;
  a.E = E;
  a.w_c = w_c;
  a.b_c = b_c;
  a.prev_tok = prev_tok;
  a.tokens = tokens;
  a.conf = conf;
  a.survival = survival;
  cudaError_t e = launch_confidence_head(*ctx, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(ctx, e, "confidence head launch");
  return DSD_OK;
}

int dsd_threshold_keep(dsd_ctx* ctx, int R, const float* conf, float threshold, int32_t* keep_len,
                       void* stream) {
  Trace trace_("dsd_threshold_keep");
  int rc = check_ctx(ctx);
  if (rc) return rc;
  if (R < 0) return fail(ctx, DSD_ERR_ARG, "R = %d < 0", R);
  if (std::isnan(threshold)) return fail(ctx, DSD_ERR_NONFINITE, "threshold is NaN");
  if (R == 0) return DSD_OK;
  if (!conf || !keep_len) return fail(ctx, DSD_ERR_ARG, "dsd_threshold_keep: NULL argument");
  cudaError_t e = launch_threshold_keep(*ctx, R, conf, threshold, keep_len,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(ctx, e, "threshold launch");
  return DSD_OK;
}

int dsd_calibration(dsd_ctx* ctx, int M, const float* conf, const int32_t* accept_len, int n_bins,
                    float* bins, float* pos, float* metrics, void* stream) {
  Trace trace_("dsd_calibration");
  int rc = check_ctx(ctx);
  if (rc) return rc;
  if (M < 0) return fail(ctx, DSD_ERR_ARG, "M = %d < 0", M);
  if (n_bins < 1 || n_bins > kMaxCalBins)
    return fail(ctx, DSD_ERR_ARG, "n_bins = %d outside 1..%d", n_bins, kMaxCalBins);
  if (!bins || !pos || !metrics) return fail(ctx, DSD_ERR_ARG, "dsd_calibration: NULL argument");
  if (M > 0 && (!conf || !accept_len)) return fail(ctx, DSD_ERR_ARG, "dsd_calibration: NULL argument");
  if ((long long)M * ctx->cfg.gamma > 0x7fffffffLL) return fail(ctx, DSD_ERR_SHAPE, "M too large");
  CalArgs a{};
  a.M = M;
  a.gamma = ctx->cfg.gamma;
  a.n_bins = n_bins;
  a.conf = conf;
  a.accept_len = accept_len;
  a.bins = bins;
  a.pos = pos;
  a.metrics = metrics;
  cudaError_t e = launch_calibration(*ctx, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(ctx, e, "calibration launch");
  return DSD_OK;
}

size_t dsd_auroc_scratch_bytes(int M, int gamma) {
  if (M < 0 || gamma < 1 || (long long)M * gamma > (1LL << 30)) return 0;
  return dsd::auroc_scratch_bytes(M, gamma);
}

int dsd_auroc(dsd_ctx* ctx, int M, const float* conf, const int32_t* accept_len, void* scratch,
              size_t scratch_bytes, double* auroc, void* stream) {
  Trace trace_("dsd_auroc");
  int rc = check_ctx(ctx);
  if (rc) return rc;
  if (M < 0) return fail(ctx, DSD_ERR_ARG, "M = %d < 0", M);
  if ((long long)M * ctx->cfg.gamma > (1LL << 30)) return fail(ctx, DSD_ERR_SHAPE, "M * gamma > 2^30");
  if (!auroc || !scratch || (M > 0 && (!conf || !accept_len)))
    return fail(ctx, DSD_ERR_ARG, "dsd_auroc: NULL argument");
  if (((uintptr_t)scratch & 255u) != 0) return fail(ctx, DSD_ERR_ALIGN, "scratch not 256-byte aligned");
  const size_t need = dsd::auroc_scratch_bytes(M, ctx->cfg.gamma);
  if (scratch_bytes < need)
    return fail(ctx, DSD_ERR_SHAPE, "scratch of %zu bytes, %zu needed", scratch_bytes, need);
  cudaError_t e = dsd::launch_auroc(*ctx, M, conf, accept_len, scratch, auroc,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(ctx, e, "auroc launch");
  return DSD_OK;
}

int dsd_propose_candidates(dsd_ctx* ctx, int R, const void* U, const void* E, const void* W,
                           const float* conf, const int32_t* prev_tok, const uint32_t* req_id,
                           float temperature, uint64_t seed, int32_t* tokens, float* lse_q,
                           float* logit_at_tok, float* survival, int32_t* cand_tok,
                           float* cand_logit, void* stream) {
  Trace trace_("dsd_propose_candidates");
  int rc = check_ctx(ctx);
  if (rc) return rc;
  if ((rc = check_R(ctx, R))) return rc;
  if ((rc = check_temperature(ctx, temperature))) return rc;
  if (R > kCandMaxR)
    return fail(ctx, DSD_ERR_CAPACITY, "R = %d > %d requests per candidate call", R, kCandMaxR);
  if (R == 0) return DSD_OK;
  if ((rc = check_table(ctx, U, "U")) || (rc = check_table(ctx, E, "E")) ||
      (rc = check_table(ctx, W, "W")))
    return rc;
  if (!conf || !prev_tok || !tokens || !lse_q || !logit_at_tok || !survival || !cand_tok ||
      !cand_logit)
    return fail(ctx, DSD_ERR_ARG, "dsd_propose_candidates: NULL argument");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ProposeArgs a{};
  a.R = R;
  a.V = ctx->cfg.V;
  a.rank = ctx->cfg.rank;
  a.gamma = ctx->cfg.gamma;
  a.dtype = ctx->cfg.dtype;
  a.act = ctx->cfg.act;
  a.bias_at_first = ctx->cfg.bias_at_first;
  a.U = U;
  a.E = E;
  a.W = W;
  a.conf = conf;
  a.prev_tok = prev_tok;
  a.req_id = req_id;
  a.temperature = temperature;
  a.seed = seed;
  a.tokens = tokens;
  a.lse_q = lse_q;
  a.logit_at_tok = logit_at_tok;
  a.survival = survival;
  a.cand_tok = cand_tok;
  a.cand_logit = cand_logit;
  // the tensor-core engine keeps the candidate lists in its repeated-rows
  // kernel (no activation); otherwise the CUDA-core engine
  cudaError_t e;
  int n_used;
  char why[256];
  if ((ctx->cfg.engine == DSD_ENGINE_TCGEN05 || auto_uses_tc(ctx, R)) &&
      ctx->cfg.act == DSD_ACT_NONE && tc_supported(*ctx, why, sizeof(why))) {
    e = launch_propose_tc(*ctx, a, s);
    n_used = tc_parts_used(*ctx, a);
    ctx->last_engine = DSD_ENGINE_TCGEN05;
  } else if (ctx->cfg.engine == DSD_ENGINE_TCGEN05) {
    return fail(ctx, DSD_ERR_UNSUPPORTED,
                "candidate sets on the tensor-core engine need no activation and its tables");
  } else {
    e = launch_propose_simt(*ctx, a, s);
    n_used = simt_grid(*ctx, a.V);
    ctx->last_engine = DSD_ENGINE_SIMT;
  }
  if (e != cudaSuccess) return cuda_fail(ctx, e, "candidate propose launch");
  e = launch_propose_finalize_n(*ctx, a, n_used, s);
  if (e == cudaSuccess) e = launch_cand_finalize(*ctx, a, n_used, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "propose finalize launch");
  return DSD_OK;
}

}  // extern "C"
