// Hardware-aware batch-global prefix scheduler ("DSpark 论文精读：置信度调度推测
// 解码、半自回归生成与大模型推理加速", section 3.2): the standalone kernel and its
// launcher.  The algorithm is in schedule.cuh.
#include "schedule.cuh"

namespace dsd {

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(SchedParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  schedule_cta(p, blockIdx.x, gridDim.x, smem);
}

SchedParams make_sched_params(const Ctx& ctx, int R, const float* survival, const float* conf,
                              const float* sps, int n_sps, int32_t* keep_len, float* theta_B) {
  SchedParams p{};
  p.survival = survival;
  p.conf = conf;
  p.sps = sps;
  p.keep_len = keep_len;
  p.theta_B = theta_B;
  p.status = ctx.ws.status;
  p.theta_bits = ctx.ws.sched_theta;
  p.order = ctx.ws.sched_order;
  p.best = ctx.ws.sched_theta + kMaxSchedItems;
  p.ticket = ctx.ws.tickets + 0;
  p.R = R;
  p.gamma = ctx.cfg.gamma;
  p.n_sps = n_sps;
  return p;
}

int schedule_ctas(const Ctx& ctx, int R) {
  // one warp per slot, at most one CTA per SM
  int grid = (R * ctx.cfg.gamma + kSchedWarps - 1) / kSchedWarps;
  return grid > ctx.num_sms ? ctx.num_sms : grid;
}

cudaError_t launch_schedule(const Ctx& ctx, int R, const float* survival, const float* sps,
                            int n_sps, int32_t* keep_len, float* theta_B, cudaStream_t s) {
  const SchedParams p = make_sched_params(ctx, R, survival, nullptr, sps, n_sps, keep_len, theta_B);
  const size_t smem = schedule_smem_bytes(R, ctx.cfg.gamma);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(schedule_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  schedule_kernel<<<schedule_ctas(ctx, R), kSchedThreads, smem, s>>>(p);
  count_launch(ctx);
  return cudaGetLastError();
}

}  // namespace dsd
