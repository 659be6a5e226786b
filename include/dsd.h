/*
 * dsd.h -- C ABI of the DSpark draft/verify hot path on one GB300 (sm_103a).
 *
 * One serving cycle for a whole batch of R requests is
 *     dsd_propose  -> dsd_schedule -> dsd_verify
 * and dsd_overlap is the separate offline-metric call.  Sources, by page title
 * and section:
 *   [TRAIN] "Qwen3.8-Flash-Next DSpark 训练实验": 评估口径/离线指标;
 *           Baseline 架构/Markov 顺序修正; Confidence head 与训练目标;
 *           Prefix reranker/候选与前缀表示
 *   [NOTES] "DSpark notes" (h.sjds.net/a/571373): 2.2 Sequential Stage;
 *           2.3 串行头的两种形态
 *   [READ]  "DSpark 论文精读：置信度调度推测解码、半自回归生成与大模型推理加速":
 *           2.2, 2.3, 3.1, 3.2, 4.1, 5
 *   [WALK]  "DeepSpec 训练全流程详解（以 Qwen3 + DSpark 为例）": 3.4 Loss,
 *           4.3 Propose, 4.4 Verify
 * dsd_loss_forward is the training-side twin: the teacher-forced DSpark loss
 * ([READ] 4.1; [WALK] 3.4).  dsd_confidence_head, dsd_threshold_keep and
 * dsd_calibration cover the scheduler's input: the confidence head, the
 * static truncation it replaces, and the calibration of its survivals.
 * dsd_propose_gated / dsd_verify_gated run the gated Markov head and
 * dsd_propose_rnn / dsd_verify_rnn the RNN head;
 * dsd_propose_candidates also returns the Markov top-16 candidate sets.
 *
 * Conventions for every call below.
 *   - Tensor arguments are DEVICE pointers owned by the caller, row-major and
 *     contiguous with the vocabulary (V) or rank (r) innermost.  The library
 *     never frees or keeps them.
 *   - Logit tables (U, P, Q) and Markov tables (E, W) use the context's dtype
 *     (DSD_BF16 or DSD_F32); all arithmetic is fp32 (fp64 for the survival
 *     products and the scheduler's running sums).
 *   - Vectorised loads need 16-byte aligned base pointers and V % 8 == 0;
 *     the Markov rank must be a multiple of 64 (or r <= 64 and a multiple of
 *     8).  Violations return DSD_ERR_ALIGN / DSD_ERR_SHAPE before any launch.
 *   - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *     default stream).  Host-detectable errors return a negative status
 *     before anything is launched; dsd_last_error() then has the message.
 *     Errors found on the device (non-finite logits or confidences, a bounded
 *     wait that ran out) are recorded in the context and returned by
 *     dsd_sync_status().  Nothing traps, asserts or aborts on the device.
 *   - No call allocates memory except dsd_create (the workspace) and the
 *     first dsd_cycle_host call (its device staging buffers).  There is no
 *     CPU fallback: without a usable sm_103a device dsd_create fails.
 *   - Calls on one context must not overlap on the GPU (the workspace is
 *     shared); use one context per concurrent stream.
 *   - temperature == 0 means greedy everywhere (draft argmax, accept iff the
 *     draft token is the target argmax, correction/bonus = target argmax).
 *   - Randomness is Philox4x32-10 (Salmon et al., SC'11) keyed by the 64-bit
 *     seed with counter (element group v/4, position, request id, stream):
 *     stream 0 draft Gumbel, 1 accept uniform, 2 residual Gumbel, 3 bonus
 *     Gumbel; u = ((w >> 9) + 0.5) * 2^-23.  Results therefore depend on the
 *     request id, never on the batch slot or the grid size.
 */
#ifndef DSD_H
#define DSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dsd_ctx dsd_ctx;

enum dsd_status {
  DSD_OK = 0,
  DSD_ERR_ARG = -1,        /* null pointer, negative size, bad enum, NaN temperature */
  DSD_ERR_ALIGN = -2,      /* pointer not 16-byte aligned, V % 8 != 0 */
  DSD_ERR_DTYPE = -3,      /* dtype not supported by the requested path */
  DSD_ERR_SHAPE = -4,      /* size outside what the context was created for */
  DSD_ERR_CUDA = -5,       /* a CUDA runtime call failed (message in dsd_last_error) */
  DSD_ERR_NONFINITE = -6,  /* device saw a non-finite logit / confidence / sum */
  DSD_ERR_TIMEOUT = -7,    /* a bounded device-side wait ran out */
  DSD_ERR_CAPACITY = -8,   /* R larger than the SPS table */
  DSD_ERR_UNSUPPORTED = -9 /* no sm_100-family device */
};

enum dsd_dtype { DSD_F32 = 0, DSD_BF16 = 1 };
enum dsd_act { DSD_ACT_NONE = 0, DSD_ACT_SILU = 1 };
/* Propose engine.  AUTO picks the 5th-generation tensor-core engine
 * (TCGEN05: TMA-staged operands, tcgen05.mma into TMEM accumulators) for bf16
 * tables and a rank that is a multiple of 64 (<= 256), at any batch size, and
 * the CUDA-core engine (SIMT) otherwise.  With an activation, and for the
 * gated and RNN heads, whose Markov representations are fp32, the tensor-core
 * engine splits each representation into hi + lo bf16 parts (|residual| <=
 * 2^-18 of the value) that two MMAs add into one fp32 accumulator.  The
 * residual pass of sampled verification runs on the tensor cores for the
 * plain head without an activation, on the CUDA cores otherwise.  MMA
 * (warp-level mma.sync tensor cores, same requirements) is only used when
 * asked for.  TCGEN05 or MMA asked for with a configuration they do not
 * support makes dsd_propose return DSD_ERR_UNSUPPORTED before any launch.
 * The tensor-core engine runs all draft steps of a call in one launch whose
 * CTAs wait for one another between steps, when the whole grid fits on the
 * device (else one launch per step, and always one per step for the gated
 * and RNN heads).  That launch is cooperative: it starts only when every CTA
 * can be resident, so calls on different streams may overlap.  The
 * environment variable DSD_PROPOSE_COOPERATIVE=0 drops the cooperative
 * attribute (for profilers that cannot replay cooperative launches); then
 * two such launches overlapping on the device can each hold SMs the other
 * needs, and their bounded waits end the calls with DSD_ERR_TIMEOUT. */
enum dsd_engine {
  DSD_ENGINE_AUTO = 0,
  DSD_ENGINE_SIMT = 1,
  DSD_ENGINE_TCGEN05 = 2,
  DSD_ENGINE_MMA = 3
};

typedef struct dsd_config {
  int V;             /* vocabulary size, multiple of 8 */
  int rank;          /* Markov rank r (256 on the pages) */
  int gamma;         /* draft positions per request (7 on the pages), 1..16 */
  int R_max;         /* largest batch a call may pass; R_max * gamma <= 4096 */
  int dtype;         /* enum dsd_dtype of U, E, W, P, Q */
  int act;           /* enum dsd_act between the two Markov tables: NONE per
                        [TRAIN] Markov 顺序修正; SILU per [READ] 2.3 */
  int bias_at_first; /* 1: position 0 is biased by E[prev_tok] ([TRAIN],
                        m_1 = W_1[D]); 0: position 0 uses U only ([READ] 2.3) */
  int engine;        /* enum dsd_engine */
  int device;        /* CUDA device ordinal the context is bound to */
} dsd_config;

/* Create a context bound to cfg->device and allocate its workspace
 * (one cudaMalloc, sized by R_max, gamma, V and the SM count).
 * Returns DSD_OK and *out, or a negative status (out untouched). */
int dsd_create(const dsd_config* cfg, dsd_ctx** out);

/* Free the workspace and the context.  NULL is accepted. */
int dsd_destroy(dsd_ctx* ctx);

/* Message of the last host-side error on this context ("" if none).  The
 * string is owned by the context and valid until the next call on it. */
const char* dsd_last_error(const dsd_ctx* ctx);

/* Wait for `stream`, then return (and clear) the device-side status of the
 * calls made so far: DSD_OK, DSD_ERR_NONFINITE or DSD_ERR_TIMEOUT. */
int dsd_sync_status(dsd_ctx* ctx, void* stream);

/* Exercise the failure path of the bounded device waits.  The pages name no
 * such call: their only failure handling is the scheduler's fallback under
 * overload ([READ] 6); this diagnostic checks the library's own rule that a
 * device wait which never completes ends in a status, not a hang.
 * One CTA runs the same bounded mbarrier waits as the tensor-core kernels on
 * barriers that nothing completes (no copy or tensor-core work is involved):
 * one waiter gives up after poll_limit polls, records DSD_ERR_TIMEOUT in the
 * context's status word and raises its CTA's abort flag; a second waiter,
 * polling with the kernels' full limit, sees the flag and stops.
 * poll_limit: 1 .. 2^20 (DSD_ERR_ARG otherwise, nothing launched).
 * roles_out: optional device int32[3] (NULL: not written): [0], [1] = 1 if
 * the first / second waiter saw its phase complete (0 expected), [2] = how
 * many of the two left their wait (2 expected).
 * After it, dsd_sync_status returns DSD_ERR_TIMEOUT (and clears it); the
 * context stays usable. */
int dsd_wait_selftest(dsd_ctx* ctx, uint32_t poll_limit, int32_t* roles_out, void* stream);

/* Bytes of device workspace held by the context. */
size_t dsd_workspace_bytes(const dsd_ctx* ctx);

/* Number of kernels this context has launched so far (host-side count of
 * every <<<>>> launch made by the calls below; memsets are not counted). */
uint64_t dsd_launch_count(const dsd_ctx* ctx);

/* Engine that ran the last dsd_propose on this context: DSD_ENGINE_SIMT,
 * DSD_ENGINE_MMA or DSD_ENGINE_TCGEN05 (DSD_ENGINE_AUTO before the first
 * call). */
int dsd_last_engine(const dsd_ctx* ctx);
/* 1 if the last dsd_cycle_host call read P in place from host memory, 0 if
 * it staged P on the device. */
int dsd_last_p_in_place(const dsd_ctx* ctx);

/*
 * dsd_gumbel_noise -- the Gumbel noise every sampled path draws from a
 * Philox word (the stream words of R5 below): out[i] = -ln(-ln u_i),
 * u_i = ((words[i] >> 9) + 0.5) * 2^-23, as the kernels compute it (the
 * hardware base-2 logarithm, and the Taylor series of -ln(1 - d) for
 * u > 15/16), so its accuracy can be checked.  words [n] u32 and out [n]
 * f32 are device pointers; asynchronous on the stream.  n < 0 or a NULL
 * pointer with n > 0 returns DSD_ERR_ARG.  Needs no context.
 */
int dsd_gumbel_noise(const uint32_t* words, float* out, int n, void* stream);

/*
 * dsd_propose -- sequential Markov-head proposal plus prefix survival.
 * [TRAIN] Markov 顺序修正; [NOTES] 2.2-2.3; [READ] 2.2, 2.3, 3.1.
 *
 * For every request r and position j = 0..gamma-1, with prev = prev_tok[r]
 * at j = 0 and the token chosen at j-1 afterwards:
 *   m      = act(E[prev, :])                  (E: [V, r] down table)
 *   b[v]   = sum_k W[v, k] * m[k]             (W: [V, r] up projection, the
 *                                              nn.Linear(r, V).weight layout)
 *   l      = U[r, j, :] + b                   (b skipped at j = 0 when
 *                                              bias_at_first == 0)
 *   T == 0: x = argmax_v l,  lse_q = logsumexp(l),   logit_at_tok = l[x]
 *   T  > 0: x = argmax_v l/T + Gumbel_v(seed, j, req, stream 0),
 *           lse_q = logsumexp(l/T),  logit_at_tok = l[x]/T
 * Argmax ties go to the lowest index.  The biased logits never reach HBM.
 *   survival[r, j] = prod_{i <= j} clamp(conf[r, i], 0, 1)   ([READ] 3.1)
 *
 * U        [R, gamma, V]  dtype        base logits of the parallel backbone
 * E, W     [V, rank]      dtype        Markov tables
 * conf     [R, gamma]     f32          per-position confidence
 * prev_tok [R]            i32          token before position 0 (anchor)
 * req_id   [R]            u32 or NULL  Philox request key (NULL: 0..R-1)
 * tokens   [R, gamma]     i32  out     draft tokens
 * lse_q    [R, gamma]     f32  out     log-normaliser of the draft softmax
 * logit_at_tok [R,gamma]  f32  out     (scaled) draft logit of each token
 * survival [R, gamma]     f32  out     prefix survival (fp64 product, rounded)
 * R == 0 is a no-op.  prev_tok outside [0, V) is DSD_ERR_ARG on the device
 * side (recorded, token 0 used) -- see dsd_sync_status.
 */
int dsd_propose(dsd_ctx* ctx, int R, const void* U, const void* E, const void* W,
                const float* conf, const int32_t* prev_tok, const uint32_t* req_id,
                float temperature, uint64_t seed, int32_t* tokens, float* lse_q,
                float* logit_at_tok, float* survival, void* stream);

/*
 * dsd_schedule -- hardware-aware batch-global prefix scheduler ([READ] 3.2).
 *
 * Maximises Theta = tau * SPS(B) with B = sum_r (1 + l_r) and
 * tau = sum_r (1 + sum_{j < l_r} survival[r, j]).  Starting from l = 0
 * (Theta = R * SPS(R)) it visits the (r, j) slots by survival descending
 * (ties: r, then j ascending), adds one slot at a time and keeps the cut with
 * the strictly largest Theta.  Because survival is non-increasing in j the
 * kept slots form a prefix of every request.
 *
 * survival [R, gamma] f32        (dsd_propose's output, values in [0, 1];
 *                                 others are clamped to [0, 1], non-finite
 *                                 ones count as 0 and set DSD_ERR_NONFINITE
 *                                 in the status word)
 * sps      [n_sps]    f32        sps[B-1] = SPS(B), steps/s at verify batch B
 * keep_len [R]        i32  out   l_r in 0..gamma
 * theta_B  [2]        f32  out   {Theta*, B*}
 * R > n_sps returns DSD_ERR_CAPACITY; slots that would push B past n_sps are
 * never taken.  The running sums are exact (integers in units of 2^-48), so
 * the cut matches an exact evaluation of Theta up to fp64 rounding of the
 * final products.
 */
int dsd_schedule(dsd_ctx* ctx, int R, const float* survival, const float* sps, int n_sps,
                 int32_t* keep_len, float* theta_B, void* stream);

/*
 * dsd_verify -- rejection verification of the kept prefixes ([WALK] 4.4;
 * [READ] 2.1, 3.1).
 *
 * P [R, gamma+1, V] holds the target logits: row t scores draft token t and
 * row keep_len[r] gives the bonus distribution.  Only rows 0..keep_len[r]
 * of each request are read.  With p_t = softmax(P[r,t]/T) and the draft
 * probability q_t(x_t) = exp(logit_at_tok - lse_q):
 *   accept x_t iff u(seed, t, req, stream 1) < min(1, p_t(x_t) / q_t(x_t)),
 *   stop at the first rejection k;
 *   k < keep_len: next_token ~ norm(max(0, p_k - q_k)) by Gumbel-max
 *                 (stream 2), where q_k is recomputed in full from U, E, W,
 *                 prev_tok and tokens; an empty residual falls back to p_k;
 *   k == keep_len: next_token ~ p_{keep_len} by Gumbel-max (stream 3).
 * T == 0: accept iff x_t == argmax P[r,t]; next_token = argmax P[r,k].
 * accept_len [R] i32 out (k), next_token [R] i32 out.  The committed tokens
 * of request r are tokens[r, :k] followed by next_token[r].
 * keep_len must come from dsd_schedule (or any values in 0..gamma; others
 * are clamped to it and set DSD_ERR_ARG in the status word); U, E, W,
 * prev_tok, lse_q, logit_at_tok may be NULL when T == 0.  Non-finite
 * values: with T == 0 a NaN in a read row sets DSD_ERR_NONFINITE; with
 * T > 0 a non-finite normaliser of a tested row does, and a NaN logit never
 * wins a Gumbel-max draw.
 */
int dsd_verify(dsd_ctx* ctx, int R, const void* P, const void* U, const void* E,
               const void* W, const int32_t* prev_tok, const int32_t* tokens,
               const float* lse_q, const float* logit_at_tok, const int32_t* keep_len,
               const uint32_t* req_id, float temperature, uint64_t seed,
               int32_t* accept_len, int32_t* next_token, void* stream);

/*
 * dsd_cycle -- dsd_propose, dsd_schedule and dsd_verify back to back on one
 * stream ([WALK] 4.2 serving loop, one iteration, whole batch).  Outputs as
 * the three calls; theta_B may be NULL.  The schedule depends on the
 * confidences only, so it runs in extra CTAs of the proposal's last launch,
 * from the survivals computed there exactly as dsd_propose computes its
 * survival output (same allocation as dsd_schedule on that output).
 * Argument errors of any of the three return before any launch.
 */
int dsd_cycle(dsd_ctx* ctx, int R, const void* U, const void* E, const void* W,
              const float* conf, const int32_t* prev_tok, const uint32_t* req_id,
              const void* P, const float* sps, int n_sps, float temperature, uint64_t seed,
              int32_t* tokens, float* lse_q, float* logit_at_tok, float* survival,
              int32_t* keep_len, float* theta_B, int32_t* accept_len, int32_t* next_token,
              void* stream);

/*
 * dsd_cycle_host -- one cycle from HOST buffers.  The per-cycle inputs
 * (U, conf, prev_tok, req_id) are copied host->device into staging buffers
 * owned by the context (allocated on the first call, sized for R_max), the
 * cycle runs, and tokens, keep_len, accept_len and next_token are copied
 * back to the host.  P is read in place when the GPU can address P_host
 * (pinned memory): verification reads only the rows the scheduler keeps,
 * so only those cross the CPU-GPU link; pageable P is staged in full.
 * dsd_last_p_in_place tells which happened.  E, W and sps are device
 * pointers (model constants resident on the GPU).  The caller must not
 * modify P_host until the call returns; the call returns after the results
 * are on the host.
 */
int dsd_cycle_host(dsd_ctx* ctx, int R, const void* U_host, const void* E, const void* W,
                   const float* conf_host, const int32_t* prev_tok_host,
                   const uint32_t* req_id_host, const void* P_host, const float* sps,
                   int n_sps, float temperature, uint64_t seed, int32_t* tokens_host,
                   int32_t* keep_len_host, int32_t* accept_len_host,
                   int32_t* next_token_host, void* stream);

/*
 * dsd_overlap -- teacher-forced offline metrics ([TRAIN] 评估口径/离线指标;
 * [READ] 3.1 overlap identity).
 *
 * For block n and valid position i < valid_len[n], with p = softmax(P[n,i]),
 * q = softmax(Q[n,i]):
 *   a[n,i]  = sum_v min(p, q),   l1[n,i] = sum_v |p - q|   (a = 1 - l1/2)
 * Invalid positions get a = l1 = 0.
 *   tau[n] = 1 + sum_i prod_{j <= i} a[n,j]
 *   accept_rate[i] = mean of a[n,i] over blocks whose position i is valid
 *   mean_tau = mean of tau over blocks with valid_len >= 1
 * (empty means are 0).
 * P_logits, Q_logits [N, gamma, V] dtype; valid_len [N] i32 in 0..gamma;
 * a, l1 [N, gamma] f32 out; tau [N] f32 out; accept_rate [gamma] f32 out;
 * mean_tau [1] f32 out.  N == 0 writes zeros to accept_rate and mean_tau.
 */
int dsd_overlap(dsd_ctx* ctx, int N, const void* P_logits, const void* Q_logits,
                const int32_t* valid_len, float* a, float* l1, float* tau,
                float* accept_rate, float* mean_tau, void* stream);

/*
 * dsd_loss_forward -- teacher-forced DSpark training loss, forward only
 * ([READ] 4.1 position-decayed L1 alignment; [WALK] 3.4 compute_dspark_loss;
 * [TRAIN] Markov 顺序修正 for the biased logits).
 *
 * Row n = b * gamma + j (block b < B, position j < gamma) has the known
 * previous token prev_tok[n] (the anchor at j = 0, the ground-truth token
 * j - 1 after it), so
 *   l      = U[b, j, :] + W E[prev_tok[n], :]     (bias skipped at j = 0 when
 *                                                  bias_at_first == 0)
 *   q = softmax(l),  p = softmax(P[b, j, :])
 *   l1[n]  = sum_v |p_v - q_v|,   accept[n] = clamp(1 - l1[n] / 2, 0, 1)
 *   ce[n]  = logsumexp(l) - l[target[n]]
 *   bce[n] = -(a log sigmoid(z) + (1 - a) log(1 - sigmoid(z))),
 *            z = conf_logit[n], a = accept[n]
 *   w_j    = exp(-j / decay) / sum_{i < gamma} exp(-i / decay)
 *   losses = { ce_loss   = sum_j w_j * mean_b ce,
 *              l1_loss   = sum_j w_j * mean_b l1,
 *              conf_loss = mean_n bce,
 *              total     = ce_alpha ce_loss + l1_alpha l1_loss + conf_alpha conf_loss }
 * The pages' defaults are decay 4, ce_alpha 0.1, l1_alpha 0.9, conf_alpha 1.
 * The biased logits never reach HBM: the bias GEMM runs on the tcgen05
 * tensor cores fused with both softmaxes, in two passes over the vocabulary
 * (normalisers, then L1); the per-row values and losses are reduced in fp64.
 *
 * U, P       [B, gamma, V]  bf16   draft base logits, target logits
 * E, W       [V, rank]      bf16   Markov tables (as dsd_propose)
 * prev_tok   [B, gamma]     i32    previous token of every row
 * target     [B, gamma]     i32    ground-truth token of every row
 * conf_logit [B, gamma]     f32    confidence-head logits
 * row_out    [4, B*gamma]   f32 out or NULL: l1, accept, ce, bce per row
 * losses     [4]            f32 out: ce_loss, l1_loss, conf_loss, total
 * Needs the tensor-core engine's configuration (bf16 tables, no activation,
 * rank a multiple of 64 up to 256), else DSD_ERR_UNSUPPORTED before any
 * launch; B <= R_max.  B == 0 writes zeros to losses.  prev_tok or target
 * outside [0, V) is DSD_ERR_ARG on the device side (recorded; the row's bias
 * is zero and its ce NaN), non-finite results DSD_ERR_NONFINITE -- see
 * dsd_sync_status.
 */
int dsd_loss_forward(dsd_ctx* ctx, int B, const void* U, const void* E, const void* W,
                     const int32_t* prev_tok, const void* P, const int32_t* target,
                     const float* conf_logit, float ce_alpha, float l1_alpha, float conf_alpha,
                     float decay, float* row_out, float* losses, void* stream);

/*
 * dsd_propose_gated -- dsd_propose with the gated Markov head ([READ] 2.3,
 * GatedMarkovHead; [NOTES] 2.3):
 *   m_j = act(E[x_{j-1}]),  g_j = sigmoid(W_g [h_j; m_j]),
 *   l_j = U_j + W (g_j * m_j)
 * and the same greedy / Gumbel selection, lse_q, logit_at_tok and survival
 * as dsd_propose.  h [R, gamma, H] (the backbone hidden states) and W_g
 * [rank, H + rank] (hidden-state columns first) in the context's dtype,
 * device, 16-byte aligned; H a positive multiple of 8.  gated_rep
 * [R, gamma, rank] f32 out: g_j * m_j per position (0 at position 0 when the
 * context has bias_at_first = 0); dsd_verify_gated reads it.  One launch for
 * the hidden-state part of every gate, then the bias steps, then the
 * finalize.  On the tensor-core engine's split mode (AUTO, TCGEN05; bf16
 * tables, rank a multiple of 64) one launch runs every draft position, its
 * CTAs computing each position's gates before its bias step; on the CUDA
 * cores (SIMT, f32) each position has a gate launch and a bias launch.
 * Errors as
 * dsd_propose; a non-finite gate argument sets DSD_ERR_NONFINITE.
 */
int dsd_propose_gated(dsd_ctx* ctx, int R, const void* U, const void* E, const void* W,
                      const void* h, int H, const void* W_g, const float* conf,
                      const int32_t* prev_tok, const uint32_t* req_id, float temperature,
                      uint64_t seed, int32_t* tokens, float* lse_q, float* logit_at_tok,
                      float* survival, float* gated_rep, void* stream);

/*
 * dsd_verify_gated -- dsd_verify for proposals of dsd_propose_gated: the
 * rejected position's draft distribution is recomputed with the gated
 * representation gated_rep [R, gamma, rank] f32 (as written by
 * dsd_propose_gated) in place of act(E[prev]).  Same arguments, outputs and
 * errors as dsd_verify otherwise; gated_rep may be NULL when temperature = 0.
 */
int dsd_verify_gated(dsd_ctx* ctx, int R, const void* P, const void* U, const void* E,
                     const void* W, const float* gated_rep, const int32_t* prev_tok,
                     const int32_t* tokens, const float* lse_q, const float* logit_at_tok,
                     const int32_t* keep_len, const uint32_t* req_id, float temperature,
                     uint64_t seed, int32_t* accept_len, int32_t* next_token, void* stream);

/*
 * dsd_propose_rnn -- dsd_propose with the RNN head ([NOTES] 2.3, its second
 * form; [READ] 2.3, RNNHead): a gated recurrent state over the drafted
 * prefix, from zero at the start of the block,
 *   m_j = act(E[x_{j-1}]),  u_j = [s_{j-1}; m_j; h_j],
 *   g = sigmoid(W_g u_j),  c = tanh(W_c u_j),  s_j = g * s_{j-1} + (1 - g) * c,
 *   o_j = tanh(W_o [s_j; m_j; h_j]),  l_j = U_j + W o_j
 * (tanh for the output nonlinearity, which the page leaves unnamed), and the
 * same greedy / Gumbel selection, lse_q, logit_at_tok and survival as
 * dsd_propose.  h [R, gamma, H] (the backbone hidden states) and W_rnn
 * [3, rank, 2 rank + H] (W_g, W_c, W_o; columns: state, Markov row, hidden
 * state) in the context's dtype, device, 16-byte aligned; H a positive
 * multiple of 8.  rnn_rep [R, gamma, rank] f32 out: o_j per position (0 at
 * position 0 when the context has bias_at_first = 0; the recursion then
 * starts at position 1); dsd_verify_rnn reads it.  One launch for the
 * hidden-state parts of all three matrices, then on the tensor-core engine
 * (split mode) one launch for all draft positions, whose CTAs compute each
 * position's state and output between the bias steps; on the CUDA cores per
 * draft position a state launch, an output launch and a bias launch; then
 * the finalize.
 * Errors as
 * dsd_propose; a non-finite gate, candidate or output argument sets
 * DSD_ERR_NONFINITE.
 */
int dsd_propose_rnn(dsd_ctx* ctx, int R, const void* U, const void* E, const void* W,
                    const void* h, int H, const void* W_rnn, const float* conf,
                    const int32_t* prev_tok, const uint32_t* req_id, float temperature,
                    uint64_t seed, int32_t* tokens, float* lse_q, float* logit_at_tok,
                    float* survival, float* rnn_rep, void* stream);

/*
 * dsd_verify_rnn -- dsd_verify for proposals of dsd_propose_rnn: the
 * rejected position's draft distribution is recomputed with o_j from
 * rnn_rep [R, gamma, rank] f32 (as written by dsd_propose_rnn).  Same
 * arguments, outputs and errors as dsd_verify otherwise; rnn_rep may be
 * NULL when temperature = 0.
 */
int dsd_verify_rnn(dsd_ctx* ctx, int R, const void* P, const void* U, const void* E,
                   const void* W, const float* rnn_rep, const int32_t* prev_tok,
                   const int32_t* tokens, const float* lse_q, const float* logit_at_tok,
                   const int32_t* keep_len, const uint32_t* req_id, float temperature,
                   uint64_t seed, int32_t* accept_len, int32_t* next_token, void* stream);

/*
 * dsd_propose_candidates -- dsd_propose plus the Markov candidate set of
 * every draft position ([TRAIN] Prefix reranker, 候选与前缀表示:
 * C_i = Top16(l_i) of the Markov-corrected scores l_i = l_i^0 + W E[t_{i-1}],
 * with this round's drafted tokens as predecessors): the set a reranker
 * scores.  Same arguments and outputs as dsd_propose, plus
 *   cand_tok [R, gamma, 16] i32 out: the 16 largest biased logits' tokens,
 *     largest first, equal logits in token order (-1 past V when V < 16)
 *   cand_logit [R, gamma, 16] f32 out: those biased logits (not divided by
 *     the temperature)
 * Runs on the tensor-core engine where dsd_propose would (AUTO, TCGEN05)
 * and the context has no activation, on the CUDA-core engine otherwise
 * (TCGEN05 with an activation is DSD_ERR_UNSUPPORTED); the biased logits
 * never reach memory: each CTA keeps per request a sorted top-16 of its
 * vocabulary tiles in shared memory, and one more launch merges the CTAs'
 * lists.  R <= 32 (DSD_ERR_CAPACITY otherwise); other errors as
 * dsd_propose.
 */
int dsd_propose_candidates(dsd_ctx* ctx, int R, const void* U, const void* E, const void* W,
                           const float* conf, const int32_t* prev_tok, const uint32_t* req_id,
                           float temperature, uint64_t seed, int32_t* tokens, float* lse_q,
                           float* logit_at_tok, float* survival, int32_t* cand_tok,
                           float* cand_logit, void* stream);

/*
 * dsd_confidence_head -- per-position confidence of the drafted tokens
 * ([TRAIN] Confidence head 与训练目标: s = w_c^T [h; m] + b_c, c = sigmoid(s),
 * with m the Markov representation W_1[t_{i-1}] before the bias projection)
 * and its prefix survival ([READ] 3.1), the scheduler's input.
 *
 *   s[r, j] = w_c[0:H] . h[r, j, :] + w_c[H:H+rank] . E[t, :] + b_c,
 *             t = prev_tok[r] at j = 0, tokens[r, j-1] after it
 *   conf[r, j] = sigmoid(s[r, j])
 *   survival[r, j] = prod_{i <= j} conf[r, i]   (fp64 product, rounded)
 * h [R, gamma, H], E [V, rank], w_c [H + rank] in the context's dtype,
 * device, 16-byte aligned; H a positive multiple of 8.  prev_tok [R],
 * tokens [R, gamma] i32 (as written by dsd_propose).  conf, survival
 * [R, gamma] f32 out.  A token outside [0, V) sets DSD_ERR_ARG in the status
 * word (row 0 of E is used); a non-finite logit sets DSD_ERR_NONFINITE (its
 * confidence is written as 0).  Host-side argument errors return before any
 * launch.  R == 0 is a no-op.  One launch.
 */
int dsd_confidence_head(dsd_ctx* ctx, int R, int H, const void* h, const void* E, const void* w_c,
                        float b_c, const int32_t* prev_tok, const int32_t* tokens, float* conf,
                        float* survival, void* stream);

/*
 * dsd_threshold_keep -- static confidence truncation, the baseline the
 * scheduler replaces ([WALK] 4.3 Propose: proposal_len = min(block, first
 * position whose confidence is below the threshold); [READ] 5 threshold
 * sweep).
 *   keep_len[r] = number of leading positions j with conf[r, j] >= threshold
 * conf [R, gamma] f32 device; keep_len [R] i32 device out.  A NaN
 * confidence ends the kept prefix; a NaN threshold is DSD_ERR_NONFINITE.
 * R == 0 is a no-op.  One launch.
 */
int dsd_threshold_keep(dsd_ctx* ctx, int R, const float* conf, float threshold, int32_t* keep_len,
                       void* stream);

/*
 * dsd_auroc -- ranking quality of predicted survival ([READ] 5: the raw
 * confidence head's AUROC, quoted beside its reliability diagram).
 *
 * conf [M, gamma] f32 and accept_len [M] i32 as for dsd_calibration.  Over
 * all M * gamma positions the score is a = prod_{i <= j} clamp(conf[r, i])
 * (fp64, the same product as dsd_calibration) and the label
 * y = (j < accept_len[r]).  *auroc (one device double) receives the
 * probability that a random positive outscores a random negative, a tie
 * counting one half (the Mann-Whitney statistic; 0.5 when a class is empty),
 * computed exactly: the positions are sorted twice (a bitonic network on
 * keys bits(a) << 1 | label) and the negatives before each positive counted.
 * scratch: caller-owned device memory of at least
 * dsd_auroc_scratch_bytes(M, gamma) bytes, 256-byte aligned (the library
 * allocates nothing); its contents are overwritten.  M * gamma <= 2^30.
 * Errors: DSD_ERR_ARG (NULL or negative M), DSD_ERR_ALIGN, DSD_ERR_SHAPE
 * (scratch too small, M * gamma too large) before any launch; accept_len
 * outside 0..gamma or a non-finite confidence set the device status.
 */
size_t dsd_auroc_scratch_bytes(int M, int gamma);
int dsd_auroc(dsd_ctx* ctx, int M, const float* conf, const int32_t* accept_len, void* scratch,
              size_t scratch_bytes, double* auroc, void* stream);

/*
 * dsd_calibration -- calibration of predicted survival against realised
 * acceptance ([READ] 3.1: per-step error and cumulative-product bias of the
 * confidence head; [READ] 5: reliability diagram, ECE).
 *
 * conf [M, gamma] f32: predicted per-step confidences (clamped to [0, 1]);
 * accept_len [M] i32 in 0..gamma: accepted prefix lengths of full-block
 * verification.  With a = prod_{i <= j} conf[r, i] (fp64) and the realised
 * survival y[r, j] = (j < accept_len[r]):
 *   bins [3][n_bins] f32 out: per reliability bin b = min(floor(a n_bins),
 *     n_bins - 1) (taken in fp64): count, mean a, mean y (0 when empty)
 *   pos [2][gamma] f32 out: mean a and mean y per position
 *   metrics [4] f32 out: ECE = sum_b count_b / (M gamma) |mean a - mean y|;
 *     abs_error = mean |conf - y| over tested positions (j <= accept_len);
 *     cumprod_bias = mean (a - y) over all positions (> 0: optimistic);
 *     the number of tested positions
 * 1 <= n_bins <= 64.  A non-finite confidence sets DSD_ERR_NONFINITE (it is
 * taken as 0), an accept_len outside 0..gamma DSD_ERR_ARG (clamped).  Uses
 * the context's workspace: calls on one context must not overlap on the
 * GPU.  M == 0 writes zeros.  One launch.
 */
int dsd_calibration(dsd_ctx* ctx, int M, const float* conf, const int32_t* accept_len, int n_bins,
                    float* bins, float* pos, float* metrics, void* stream);

/*
 * dsd_propose_noalloc -- dsd_propose for callers that cannot allocate device
 * memory.  The paper has no counterpart: this is a library convenience.
 *
 * Some callers cannot call cudaMalloc: an inference engine that hands all of
 * device memory to its own pool at start-up and forbids plugins to allocate,
 * or a latency-critical loop that must not pay an allocation's implicit
 * synchronisation.  They cannot create a dsd_ctx, whose workspace is
 * allocated, so this call takes the configuration fields directly (their
 * meaning and limits as in dsd_config) and runs dsd_propose's CUDA-core
 * engine on the current device.  It drafts the same tokens as dsd_propose
 * with engine DSD_ENGINE_SIMT; on devices with at most 256 SMs it splits the
 * vocabulary the same way and its lse_q / logit_at_tok are the same values,
 * beyond that they agree within the parity tolerance (1e-4).
 *
 * Its scratch (status word, argmax keys and log-sum-exp partials, about
 * 4.2 MB) is a fixed-size array in the library's device memory, held by
 * every GPU that loads the library until the process exits.  Limits:
 * R * gamma <= 1024; larger calls return DSD_ERR_SHAPE without launching
 * anything.  The call allocates nothing (no cudaMalloc, cudaFree or
 * allocating library routine).  All calls on a device share that array and
 * each call leaves its contents behind; the parts that must start at zero
 * are cleared at the start of every call.  Calls whose executions overlap on
 * the GPU (other streams, other host threads) race on the array: serialise
 * them.  The first call on a device looks up the array's device address
 * with that device current and caches it for the process; make that first
 * call before any stream capture.  The cached address does not survive
 * cudaDeviceReset.
 *
 * status: optional device pointer to one int32 (NULL: not reported).  After
 * the call's kernels it receives, in stream order, the device-side status of
 * this call: DSD_OK, DSD_ERR_ARG (a prev_tok outside [0, V), drafted from
 * token 0 instead) or DSD_ERR_NONFINITE (a non-finite logit or confidence).
 */
int dsd_propose_noalloc(int V, int rank, int gamma, int dtype, int act, int bias_at_first,
                        int R, const void* U, const void* E, const void* W, const float* conf,
                        const int32_t* prev_tok, const uint32_t* req_id, float temperature,
                        uint64_t seed, int32_t* tokens, float* lse_q, float* logit_at_tok,
                        float* survival, int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSD_H */
