// Internal declarations shared by the C-ABI layer and the kernel files.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime.h>

namespace dsd {

constexpr int kActNone = 0;
constexpr int kActSilu = 1;

constexpr int kMaxGamma = 16;
constexpr int kMaxCalBins = 64;      // reliability bins of dsd_calibration
constexpr int kCandK = 16;           // Markov candidate set size (top-16)
constexpr int kCandMaxR = 32;        // requests per call of dsd_propose_candidates
constexpr int kGateZhFactor = 12;    // gated / RNN heads: split-K partials, 12 x R_max gamma x rank floats
constexpr int kMaxSchedItems = 4096;  // R_max * gamma
constexpr int kVerifySplits = 8;      // V chunks per verified row
constexpr int kStepSyncWords = 64;    // kMaxGamma counters + an abort word, padded to 32,
                                       // then 2 per position for a head's step phases

// Status codes (mirror enum dsd_status in include/dsd.h).
constexpr int kOk = 0;
constexpr int kErrArg = -1;
constexpr int kErrNonfinite = -6;
constexpr int kErrTimeout = -7;

// Partial result of one CTA over a slice of the vocabulary for one row:
// the online log-sum-exp state (base 2) and a packed argmax key.
struct RowPart {
  float m, s;
  unsigned long long key;
};

// Device workspace, carved out of one allocation at context creation.
struct Workspace {
  int* status;                  // first device-side error of the calls so far
  unsigned int* counters;       // [16] tickets / barrier counters (zeroed per call)
  unsigned long long* keys;     // [gamma][R_max] argmax keys of the propose steps
  unsigned int* step_sync;      // [kStepSyncWords], right after keys (one memset clears both):
                                // per-position counters of a several-position propose launch
  float2* lse_parts;            // [gamma][n_part][R_max] (m, s) partials
  RowPart* vparts;              // [R_max*(gamma+1)][kVerifySplits]
  int* rej_list;                // [R_max] requests with a rejection (sampled verify)
  int* rej_k;                   // [R_max] rejection position per request
  float* rej_lseP;              // [R_max] target log-normaliser at the rejected row
  unsigned long long* res_keys; // [2][R_max] residual key, fallback key
  float* res_sums;              // [2][R_max] sum of the residual, sum of p
  float* ov_parts;              // scratch of the overlap kernels
  unsigned long long* sched_theta;  // [kMaxSchedItems + 1] Theta bits per cut; last: their maximum
  int* sched_order;             // [kMaxSchedItems] slot at each position of the schedule order
  unsigned int* tickets;        // [64] last-CTA tickets; each user resets its own to zero
  float4* loss_parts1;          // [num_sms][R_max*gamma] log-sum-exp partials of the loss
  float* loss_parts2;           // [num_sms][R_max*gamma] L1 partials of the loss
  float* loss_ltgt;             // [R_max*gamma] draft logit at the target token
  double* loss_red;             // [64][3] per-CTA sums of the loss finalize
  double* cal_acc;              // [2 kMaxCalBins + 2 + 2 kMaxGamma] calibration sums (zero between calls)
  unsigned long long* cal_cnt;  // [kMaxCalBins + 1] calibration counts (zero between calls)
  float* gate_zh;               // split-K partials of the gated / RNN heads' hidden-state parts
  float* rnn_state;             // [2][R_max][rank] RNN head state, ping-pong over the draft steps
  unsigned long long* cand_parts;  // [gamma][n_part][min(R_max, kCandMaxR)][kCandK] candidate keys
};

struct Config {
  int V, rank, gamma, R_max, dtype, act, bias_at_first, engine, device;
};

struct Ctx {
  Config cfg;
  int num_sms;
  int n_part;                  // CTAs of a propose step (lse partial slots)
  void* ws_base;
  size_t ws_bytes;
  Workspace ws;
  // host-buffer staging for dsd_cycle_host (allocated on first use)
  void* stage_base;
  size_t stage_bytes;
  char err[512];
  mutable unsigned long long launches;  // kernels launched by this context
  int last_engine;                      // engine of the last propose (enum dsd_engine)
  int last_p_in_place;                  // dsd_cycle_host: 1 if P was read in place from host memory
};

inline void count_launch(const Ctx& c, int n = 1) { c.launches += (unsigned long long)n; }

// ----------------------------------------------------------------- launchers
struct ProposeArgs {
  int R, V, rank, gamma, dtype, act, bias_at_first;
  const void* U;
  const void* E;
  const void* W;
  const float* conf;
  const int32_t* prev_tok;
  const uint32_t* req_id;
  float temperature;
  uint64_t seed;
  int32_t* tokens;
  float* lse_q;
  float* logit_at_tok;
  float* survival;
  // gated Markov head (gate_h == nullptr: the plain head)
  const void* gate_h;   // [R, gamma, H] backbone hidden states
  const void* W_g;      // [rank, H + rank]
  int H;
  float* gated_rep;     // [R, gamma, rank] f32 out: g * m per position (o_j for the RNN head)
  // RNN head (rnn_W != nullptr; gate_h, H and gated_rep then hold its hidden
  // states, their width and its per-position output o_j)
  const void* rnn_W;    // [3, rank, 2 rank + H]: W_g, W_c, W_o
  // Markov candidate sets (cand_tok == nullptr: none)
  int32_t* cand_tok;    // [R, gamma, kCandK]
  float* cand_logit;    // [R, gamma, kCandK]
  // the schedule of the whole cycle, run by extra CTAs of the finalize
  // (sched_keep == nullptr: none)
  const float* sched_sps;
  int sched_n_sps;
  int32_t* sched_keep;
  float* sched_theta;
};
cudaError_t launch_cand_finalize(const Ctx& ctx, const ProposeArgs& a, int n_used, cudaStream_t s);

cudaError_t launch_propose_simt(const Ctx& ctx, const ProposeArgs& a, cudaStream_t s);
cudaError_t launch_gate_h(const Ctx& ctx, const ProposeArgs& a, cudaStream_t s);
struct HeadStepParams;
// The per-step head arguments of a gated or RNN proposal (head_step.cuh).
HeadStepParams head_step_params(const Ctx& ctx, const ProposeArgs& a);
cudaError_t launch_gate_step(const Ctx& ctx, const ProposeArgs& a, int j, cudaStream_t s);
cudaError_t launch_rnn_h(const Ctx& ctx, const ProposeArgs& a, cudaStream_t s);
cudaError_t launch_rnn_step(const Ctx& ctx, const ProposeArgs& a, int j, cudaStream_t s);
cudaError_t launch_propose_tc(const Ctx& ctx, const ProposeArgs& a, cudaStream_t s);
cudaError_t launch_propose_mma(const Ctx& ctx, const ProposeArgs& a, cudaStream_t s);
int mma_vranges(const Ctx& ctx, int R);
cudaError_t launch_propose_finalize(const Ctx& ctx, const ProposeArgs& a, cudaStream_t s);

cudaError_t launch_schedule(const Ctx& ctx, int R, const float* survival, const float* sps,
                            int n_sps, int32_t* keep_len, float* theta_B, cudaStream_t s);

struct VerifyArgs {
  int R, V, rank, gamma, dtype, act, bias_at_first;
  const float* gated_rep;   // gated head: [R, gamma, rank] representations (else nullptr)
  const void* P;
  const void* U;
  const void* E;
  const void* W;
  const int32_t* prev_tok;
  const int32_t* tokens;
  const float* lse_q;
  const float* logit_at_tok;
  const int32_t* keep_len;
  const uint32_t* req_id;
  float temperature;
  uint64_t seed;
  int32_t* accept_len;
  int32_t* next_token;
};

cudaError_t launch_verify(const Ctx& ctx, const VerifyArgs& a, cudaStream_t s);

struct OverlapArgs {
  int N, V, gamma, dtype;
  const void* P;
  const void* Q;
  const int32_t* valid_len;
  float* a;
  float* l1;
  float* tau;
  float* accept_rate;
  float* mean_tau;
};

cudaError_t launch_overlap(const Ctx& ctx, const OverlapArgs& a, cudaStream_t s);

struct ConfHeadArgs {
  int R, H, V, rank, gamma, dtype;
  const void* h;
  const void* E;
  const void* w_c;
  float b_c;
  const int32_t* prev_tok;
  const int32_t* tokens;
  float* conf;
  float* survival;
};
cudaError_t launch_confidence_head(const Ctx& ctx, const ConfHeadArgs& a, cudaStream_t s);
cudaError_t launch_threshold_keep(const Ctx& ctx, int R, const float* conf, float threshold,
                                  int32_t* keep_len, cudaStream_t s);
struct CalArgs {
  int M, gamma, n_bins;
  const float* conf;
  const int32_t* accept_len;
  float* bins;
  float* pos;
  float* metrics;
};
cudaError_t launch_calibration(const Ctx& ctx, const CalArgs& a, cudaStream_t s);
size_t auroc_scratch_bytes(int M, int gamma);
cudaError_t launch_auroc(const Ctx& ctx, int M, const float* conf, const int32_t* accept_len,
                         void* scratch, double* auroc, cudaStream_t s);

struct LossArgs {
  int B, V, rank, gamma, bias_at_first;
  const void* U;
  const void* E;
  const void* W;
  const void* P;
  const int32_t* prev_tok;
  const int32_t* target;
  const float* conf_logit;
  double ce_alpha, l1_alpha, conf_alpha, decay;
  float* row_out;
  float* losses;
};

cudaError_t launch_loss(const Ctx& ctx, const LossArgs& a, cudaStream_t s);

// Self-test of the bounded mbarrier waits (wait_selftest.cu).
cudaError_t launch_wait_selftest(const Ctx& ctx, uint32_t poll_limit, int32_t* roles_out,
                                 cudaStream_t s);

// Swizzle mask for 16-byte chunks of a staged table row (see propose_simt.cu).
inline int chunk_swizzle_mask(int chunks_per_row) {
  if (chunks_per_row % 8 == 0) return 7;
  if ((chunks_per_row & (chunks_per_row - 1)) == 0) return chunks_per_row - 1;
  return 0;
}

}  // namespace dsd
