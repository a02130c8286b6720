// fa_static.cu -- the split-KV forward for callers that cannot allocate.
//
// Some callers of this library cannot call cudaMalloc: a plugin hosted by an
// application that hands out all device memory through its own pool (a raw
// cudaMalloc would bypass that pool's accounting, or fail once the pool has
// reserved the device), or a latency-critical path that cannot afford
// cudaMalloc's implicit device-wide synchronisation.  fa_fwd_split needs a
// scratch workspace from its caller; fa_fwd_split_static instead uses the
// fixed array below, which every GPU that loads this library holds until the
// process exits.
#include <mutex>

#include "fa_internal.h"

namespace fa {

// Scratch of the static split-KV entry point: the fp32 partial outputs and
// log-sum-exps of all splits (split_workspace_bytes(...) of it per call).
constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_split_scratch[kStaticScratchBytes];

// In host code g_split_scratch names a host-side stand-in, not device memory:
// the device address comes from cudaGetSymbolAddress, once per device, with
// that device current.
static void* g_scratch_addr[64] = {nullptr};
static std::mutex g_scratch_mu;

static fa_status static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= 64) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_split_scratch);
    if (e != cudaSuccess) return cuda_status(e);
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FA_OK;
}

}  // namespace fa

extern "C" fa_status fa_fwd_split_static(const void* q, const void* k, const void* v, void* o,
                                         float* lse, int B, int Hq, int Hkv, int T, int d,
                                         float scale, int causal, fa_dtype dtype, int num_splits,
                                         void* stream) {
  fa::FwdArgs a{q, k, v, o, lse, B, Hq, Hkv, T, d, scale, causal, dtype,
                static_cast<cudaStream_t>(stream)};
  fa_status s = fa::validate_fwd(a);
  if (s != FA_OK) return s;
  if (num_splits < 1 || num_splits > fa::kMaxSplits) return FA_ERR_INVALID_ARG;
  if (dtype == FA_DTYPE_F32) return fa::launch_simt(a);
  if (num_splits == 1) return fa::launch_tc(a);
  const size_t need = fa::split_workspace_bytes(B, Hq, T, d, num_splits);
  if (need > fa::kStaticScratchBytes) return FA_ERR_WORKSPACE;
  void* scratch = nullptr;
  s = fa::static_scratch(&scratch);
  if (s != FA_OK) return s;
  // every partial the merge reads is written by the same call, so nothing in
  // the scratch needs clearing first
  return fa::launch_tc_split(a, num_splits, scratch, fa::kStaticScratchBytes);
}
