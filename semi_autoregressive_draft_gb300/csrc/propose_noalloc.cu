// dsd_propose_noalloc: the propose call for callers that must not allocate
// device memory.
//
// Who needs it: code that may not call cudaMalloc once it runs, e.g. a
// serving engine that hands all of device memory to its own pool at start-up
// and does not let plugins allocate, or a latency-critical loop that must
// not risk an allocation's implicit device synchronisation.  Such callers
// cannot create a dsd_ctx (dsd_create allocates the workspace), so this
// entry point takes the configuration directly and keeps its scratch (the
// status word, the per-step argmax keys and the per-CTA log-sum-exp
// partials) in a fixed-size array in the library's own device memory, which
// every GPU that loads the library holds until the process exits.
//
// It runs the CUDA-core propose engine.  Sizes: R * gamma <= 1024 and at most
// 512 CTAs per draft step (twice the SM count up to 256 SMs, the split the
// context call uses); larger R * gamma is rejected with DSD_ERR_SHAPE.
// All calls on a device share the one array and each call leaves its
// contents behind: the status word and the argmax keys are cleared at the
// start of every call, and calls whose executions overlap on the GPU
// (different streams, or concurrent host threads) race on the array and
// must be serialised by the caller.  The first call on a device looks up the
// array's device address (cudaGetSymbolAddress, with that device current)
// and caches it for the life of the process; make that first call before
// any stream capture.  The cache does not survive cudaDeviceReset.
#include <mutex>
#include <string.h>

#include <nvtx3/nvToolsExt.h>

#include "../../include/dsd.h"
#include "dsd_internal.h"

namespace dsd {
int simt_grid(const Ctx& ctx, int V);
cudaError_t launch_propose_finalize_n(const Ctx& ctx, const ProposeArgs& a, int n_used,
                                      cudaStream_t s);
}  // namespace dsd

namespace {

constexpr int kNoallocMaxItems = 1024;  // R * gamma
constexpr int kNoallocMaxParts = 512;   // CTAs of one propose step
constexpr size_t kStatusBytes = 256;
constexpr size_t kKeysBytes = sizeof(unsigned long long) * (size_t)kNoallocMaxItems;
constexpr size_t kPartsBytes = sizeof(float2) * (size_t)kNoallocMaxItems * kNoallocMaxParts;
constexpr size_t kScratchBytes = kStatusBytes + kKeysBytes + kPartsBytes;  // ~4.2 MB

struct DeviceScratch {
  bool ready;
  unsigned char* base;  // device address of the array on this device
  int num_sms;
  int major;
};

constexpr int kMaxDevices = 64;
DeviceScratch g_devices[kMaxDevices];
std::mutex g_mutex;

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

// Once per device, with that device current: the array's device address.
int scratch_for_current_device(DeviceScratch* out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return DSD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceScratch& d = g_devices[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return DSD_ERR_CUDA;
    int sms = 0, major = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
      return DSD_ERR_CUDA;
    d.base = static_cast<unsigned char*>(p);
    d.num_sms = sms;
    d.major = major;
    d.ready = true;
  }
  *out = d;
  return DSD_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

static int propose_noalloc_impl(int V, int rank, int gamma, int dtype, int act, int bias_at_first,
                                int R, const void* U, const void* E, const void* W,
                                const float* conf, const int32_t* prev_tok, const uint32_t* req_id,
                                float temperature, uint64_t seed, int32_t* tokens, float* lse_q,
                                float* logit_at_tok, float* survival, int32_t* status,
                                void* stream);

extern "C" int dsd_propose_noalloc(int V, int rank, int gamma, int dtype, int act,
                                   int bias_at_first, int R, const void* U, const void* E,
                                   const void* W, const float* conf, const int32_t* prev_tok,
                                   const uint32_t* req_id, float temperature, uint64_t seed,
                                   int32_t* tokens, float* lse_q, float* logit_at_tok,
                                   float* survival, int32_t* status, void* stream) {
  nvtxRangePushA("dsd_propose_noalloc");
  const int rc = propose_noalloc_impl(V, rank, gamma, dtype, act, bias_at_first, R, U, E, W, conf,
                                      prev_tok, req_id, temperature, seed, tokens, lse_q,
                                      logit_at_tok, survival, status, stream);
  nvtxRangePop();
  return rc;
}

static int propose_noalloc_impl(int V, int rank, int gamma, int dtype, int act, int bias_at_first,
                                int R, const void* U, const void* E, const void* W,
                                const float* conf, const int32_t* prev_tok, const uint32_t* req_id,
                                float temperature, uint64_t seed, int32_t* tokens, float* lse_q,
                                float* logit_at_tok, float* survival, int32_t* status,
                                void* stream) {
  if (V < 8 || V % 8 != 0) return DSD_ERR_ALIGN;
  const bool rank_ok = (rank % 64 == 0 && rank <= 256) || (rank > 0 && rank <= 64 && rank % 8 == 0);
  if (!rank_ok || gamma < 1 || gamma > dsd::kMaxGamma || R < 0) return DSD_ERR_SHAPE;
  if ((long long)R * gamma > kNoallocMaxItems) return DSD_ERR_SHAPE;
  if (dtype != DSD_F32 && dtype != DSD_BF16) return DSD_ERR_DTYPE;
  if (act != DSD_ACT_NONE && act != DSD_ACT_SILU) return DSD_ERR_ARG;
  if (!(temperature >= 0.f) || temperature > 3.0e38f) return DSD_ERR_ARG;
  if (R == 0) return DSD_OK;
  if (!U || !E || !W || !conf || !prev_tok || !tokens || !lse_q || !logit_at_tok || !survival)
    return DSD_ERR_ARG;
  if (!aligned16(U) || !aligned16(E) || !aligned16(W)) return DSD_ERR_ALIGN;

  DeviceScratch d;
  int rc = scratch_for_current_device(&d);
  if (rc != DSD_OK) return rc;
  if (d.major != 10) return DSD_ERR_UNSUPPORTED;

  // A context description that points into the static array; nothing here
  // owns memory.
  dsd::Ctx c;
  memset(&c, 0, sizeof(c));
  int dev = 0;
  cudaGetDevice(&dev);
  c.cfg = dsd::Config{V, rank, gamma, R, dtype, act, bias_at_first ? 1 : 0, DSD_ENGINE_SIMT, dev};
  c.num_sms = d.num_sms;
  c.n_part = 2 * d.num_sms < kNoallocMaxParts ? 2 * d.num_sms : kNoallocMaxParts;
  c.ws.status = reinterpret_cast<int*>(d.base);
  c.ws.keys = reinterpret_cast<unsigned long long*>(d.base + kStatusBytes);
  c.ws.lse_parts = reinterpret_cast<float2*>(d.base + kStatusBytes + kKeysBytes);

  dsd::ProposeArgs a{};
  a.R = R;
  a.V = V;
  a.rank = rank;
  a.gamma = gamma;
  a.dtype = dtype;
  a.act = act;
  a.bias_at_first = bias_at_first ? 1 : 0;
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

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(c.ws.status, 0, sizeof(int), s) != cudaSuccess) return DSD_ERR_CUDA;
  if (dsd::launch_propose_simt(c, a, s) != cudaSuccess) return DSD_ERR_CUDA;
  if (dsd::launch_propose_finalize_n(c, a, dsd::simt_grid(c, V), s) != cudaSuccess)
    return DSD_ERR_CUDA;
  // the call's device status, copied in stream order (no allocation)
  if (status && cudaMemcpyAsync(status, c.ws.status, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                                s) != cudaSuccess)
    return DSD_ERR_CUDA;
  return DSD_OK;
}
