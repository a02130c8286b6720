// fa_bwd_tc.cu -- attention backward on the tensor cores (bf16 / fp16).
#include "fa_internal.h"

namespace fa {

static __device__ unsigned int g_bwd_err;

bool bwd_tc_supported(const BwdArgs& a) {
  (void)a;
  return false;
}

fa_status launch_bwd_tc(const BwdArgs& a) {
  (void)a;
  return FA_ERR_UNSUPPORTED;
}

fa_status bwd_read_and_clear_error(unsigned int* word) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_bwd_err, sizeof(v));
  if (e != cudaSuccess) return cuda_status(e);
  if (v) {
    e = cudaMemcpyToSymbol(g_bwd_err, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_status(e);
  }
  *word = v;
  return FA_OK;
}

}  // namespace fa
