// tcgen05 path of the Markov-head bias projection (not built yet).
#include <stdio.h>

#include "dsd_common.cuh"

namespace dsd {

int tc_supported(const Ctx&, char* why, size_t why_len) {
  snprintf(why, why_len, "tcgen05 propose engine not available in this build");
  return 0;
}

int tc_grid(const Ctx& ctx) { return ctx.num_sms; }

cudaError_t launch_propose_tc(const Ctx&, const ProposeArgs&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace dsd
