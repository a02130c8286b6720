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
// the device address comes from cudaGetSymbolAddress, with that device
// current.  The look-up is done once per device and CUDA context: the cache
// also holds the id of the context it was made in (cuCtxGetId, unique for the
// life of the process), so that after a cudaDeviceReset, which unloads the
// module and can move the array, the next call looks the address up again
// instead of handing the kernels a stale pointer.
struct ScratchSlot {
  void* addr = nullptr;
  unsigned long long ctx_id = 0;
};
static ScratchSlot g_scratch_slot[64];
static std::mutex g_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// id of the calling thread's current context (0 when none is current yet or
// the driver does not export the calls)
static unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool resolved = false;
  if (!resolved) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) ==
            cudaSuccess && q1 == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) ==
            cudaSuccess && q2 == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f2);
    resolved = true;
  }
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

static fa_status static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= 64) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchSlot& slot = g_scratch_slot[dev];
  const unsigned long long id = current_ctx_id();
  if (slot.addr == nullptr || id == 0 || id != slot.ctx_id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_split_scratch);
    if (e != cudaSuccess) {
      slot.addr = nullptr;
      return cuda_status(e);
    }
    slot.addr = p;
    // the look-up made the device's primary context current if none was
    slot.ctx_id = id != 0 ? id : current_ctx_id();
  }
  *out = slot.addr;
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
