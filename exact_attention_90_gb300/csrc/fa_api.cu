// fa_api.cu -- the C ABI of libfa.so: argument checks, tensor maps, dispatch.
//
// Entry points are declared (with their contracts) in include/fa.h and
// include/fa_unit.h.  Nothing here allocates device memory or synchronises on
// the fa_fwd path; errors are returned before anything is enqueued.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "fa_internal.h"

namespace fa {

fa_status tc_read_and_clear_error(unsigned int* word);    // fa_tc.cu
fa_status unit_read_and_clear_error(unsigned int* word);  // fa_unit.cu

static thread_local int t_last_cuda_error = 0;

fa_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return FA_OK;
  t_last_cuda_error = static_cast<int>(e);
  return FA_ERR_CUDA;
}

fa_status cu_status(CUresult r) {
  if (r == CUDA_SUCCESS) return FA_OK;
  t_last_cuda_error = static_cast<int>(r);
  return FA_ERR_CUDA;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

fa_status validate_fwd(const FwdArgs& a) {
  if (!a.q || !a.k || !a.v || !a.o || !a.lse) return FA_ERR_INVALID_ARG;
  if (a.B <= 0 || a.Hq <= 0 || a.Hkv <= 0 || a.T <= 0 || a.d <= 0) return FA_ERR_INVALID_ARG;
  if (a.T >= (1 << 30)) return FA_ERR_INVALID_ARG;  // band arithmetic stays in 32 bits
  if (a.Hq % a.Hkv != 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(a.scale)) return FA_ERR_INVALID_ARG;
  if (a.causal != 0 && a.causal != 1) return FA_ERR_INVALID_ARG;
  if (a.dtype != FA_DTYPE_F32 && a.dtype != FA_DTYPE_BF16 && a.dtype != FA_DTYPE_F16)
    return FA_ERR_UNSUPPORTED;
  if (a.d != 16 && a.d != 32 && a.d != 64 && a.d != 128) return FA_ERR_UNSUPPORTED;
  // sizes: element counts must fit comfortably in 63 bits and the grid in 2^31
  const double eq = static_cast<double>(a.B) * a.Hq * a.T * a.d;
  if (eq > 9.0e15) return FA_ERR_INVALID_ARG;
  const double units = static_cast<double>(a.B) * a.Hq * ((a.T + 63) / 64);
  if (units > 2.0e9) return FA_ERR_INVALID_ARG;
  if (static_cast<double>(a.B) * a.Hq > 2.0e9 || static_cast<double>(a.B) * a.Hkv > 2.0e9)
    return FA_ERR_INVALID_ARG;
  if (!aligned16(a.q) || !aligned16(a.k) || !aligned16(a.v) || !aligned16(a.o) ||
      !aligned16(a.lse))
    return FA_ERR_MISALIGNED;
  const size_t e = a.dtype == FA_DTYPE_F32 ? 4 : 2;
  const size_t nq = static_cast<size_t>(a.B) * a.Hq * a.T * a.d * e;
  const size_t nkv = static_cast<size_t>(a.B) * a.Hkv * a.T * a.d * e;
  const size_t nl = static_cast<size_t>(a.B) * a.Hq * a.T * 4;
  if (overlap(a.o, nq, a.q, nq) || overlap(a.o, nq, a.k, nkv) || overlap(a.o, nq, a.v, nkv) ||
      overlap(a.o, nq, a.lse, nl) || overlap(a.lse, nl, a.q, nq) || overlap(a.lse, nl, a.k, nkv) ||
      overlap(a.lse, nl, a.v, nkv))
    return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// ---------------------------------------------------------------- tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static CUresult g_encode_status = CUDA_ERROR_NOT_INITIALIZED;
static std::once_flag g_encode_once;

static void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
    g_encode_status = CUDA_ERROR_NOT_FOUND;
    return;
  }
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  g_encode_status = CUDA_SUCCESS;
}

CUresult make_tmap_16bit(CUtensorMap* map, const void* base, int d, int T, long long BH,
                         int box_x, int swizzle, bool f16, int box_rows) {
  std::call_once(g_encode_once, load_encode);
  if (g_encode_status != CUDA_SUCCESS) return g_encode_status;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(T) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_x), static_cast<cuuint32_t>(box_rows), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  return g_encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  static_cast<CUtensorMapSwizzle>(swizzle), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

fa_status read_and_clear_device_error(cudaStream_t stream, unsigned int* word) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_status(e);
  unsigned int a = 0, b = 0;
  fa_status s = tc_read_and_clear_error(&a);
  if (s != FA_OK) return s;
  s = unit_read_and_clear_error(&b);
  if (s != FA_OK) return s;
  unsigned int c = 0;
  s = bwd_read_and_clear_error(&c);
  if (s != FA_OK) return s;
  *word = a | b | c;
  return FA_OK;
}

}  // namespace fa

// ---------------------------------------------------------------- C ABI
extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                 int Hkv, int T, int d, float scale, int causal, fa_dtype dtype, void* stream) {
  fa::FwdArgs a{q, k, v, o, lse, B, Hq, Hkv, T, d, scale, causal, dtype,
                static_cast<cudaStream_t>(stream)};
  fa_status s = fa::validate_fwd(a);
  if (s != FA_OK) return s;
  return dtype == FA_DTYPE_F32 ? fa::launch_simt(a) : fa::launch_tc(a);
}

fa_status fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int Hq, int Hkv, int T, int d, float scale, int window_left,
                        int window_right, fa_dtype dtype, void* stream) {
  fa::FwdArgs a{q, k, v, o, lse, B, Hq, Hkv, T, d, scale, 0, dtype,
                static_cast<cudaStream_t>(stream)};
  if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
  a.window_left = window_left;
  a.window_right = window_right;
  fa_status s = fa::validate_fwd(a);
  if (s != FA_OK) return s;
  return dtype == FA_DTYPE_F32 ? fa::launch_simt(a) : fa::launch_tc(a);
}

fa_status fa_fwd_local_global(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int Hq, int Hkv, int T, int d, float scale, int causal,
                             int local_window, const int* global_tokens, int num_global,
                             fa_dtype dtype, void* workspace, unsigned long long workspace_bytes,
                             void* stream) {
  fa::FwdArgs a{q, k, v, o, lse, B, Hq, Hkv, T, d, scale, causal, dtype,
                static_cast<cudaStream_t>(stream)};
  if (local_window < 0 || num_global < 0) return FA_ERR_INVALID_ARG;
  if (num_global > 0 && global_tokens == nullptr) return FA_ERR_INVALID_ARG;
  a.window_left = local_window;
  a.window_right = local_window;
  fa_status s = fa::validate_fwd(a);
  if (s != FA_OK) return s;
  if (reinterpret_cast<uintptr_t>(global_tokens) & 3u) return FA_ERR_MISALIGNED;
  if (workspace == nullptr) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 15u) return FA_ERR_MISALIGNED;
  const size_t lg_need = fa::lg_workspace_bytes(T);
  if (workspace_bytes < lg_need) return FA_ERR_WORKSPACE;
  const size_t e = dtype == FA_DTYPE_F32 ? 4 : 2;
  // packed global keys when the workspace has room (16-bit inputs only)
  const size_t pack = dtype == FA_DTYPE_F32 ? 0 : fa::lg_pack_workspace_bytes(B, Hkv, d, e, num_global);
  const bool packed = dtype != FA_DTYPE_F32 && num_global > 0 && workspace_bytes >= lg_need + pack;
  const size_t need = lg_need + (packed ? pack : 0);
  const size_t nq = static_cast<size_t>(B) * Hq * T * d * e;
  const size_t nkv = static_cast<size_t>(B) * Hkv * T * d * e;
  const size_t nl = static_cast<size_t>(B) * Hq * T * 4;
  const size_t ng = static_cast<size_t>(num_global) * 4;
  if (fa::overlap(workspace, need, q, nq) || fa::overlap(workspace, need, k, nkv) ||
      fa::overlap(workspace, need, v, nkv) || fa::overlap(workspace, need, o, nq) ||
      fa::overlap(workspace, need, lse, nl) ||
      (ng > 0 && (fa::overlap(workspace, need, global_tokens, ng) ||
                  fa::overlap(o, nq, global_tokens, ng) || fa::overlap(lse, nl, global_tokens, ng))))
    return FA_ERR_INVALID_ARG;
  s = fa::launch_lg_prep(a, global_tokens, num_global, workspace);
  if (s != FA_OK) return s;
  if (packed) {
    s = fa::launch_lg_pack(a, num_global, static_cast<uint8_t*>(workspace) + lg_need);
    if (s != FA_OK) return s;
  }
  return dtype == FA_DTYPE_F32 ? fa::launch_simt(a) : fa::launch_tc(a);
}

unsigned long long fa_fwd_local_global_workspace_size(int T) {
  if (T <= 0) return 0;
  return fa::lg_workspace_bytes(T);
}

unsigned long long fa_fwd_local_global_packed_workspace_size(int B, int Hkv, int T, int d,
                                                             fa_dtype dtype, int num_global) {
  if (B <= 0 || Hkv <= 0 || T <= 0 || d <= 0 || num_global < 0) return 0;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F16 && dtype != FA_DTYPE_F32) return 0;
  const size_t lg = fa::lg_workspace_bytes(T);
  if (dtype == FA_DTYPE_F32 || num_global == 0) return lg;
  return lg + fa::lg_pack_workspace_bytes(B, Hkv, d, 2, num_global);
}

fa_status fa_fwd_simt(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int Hq, int Hkv, int T, int d, float scale, int causal, fa_dtype dtype,
                      void* stream) {
  fa::FwdArgs a{q, k, v, o, lse, B, Hq, Hkv, T, d, scale, causal, dtype,
                static_cast<cudaStream_t>(stream)};
  fa_status s = fa::validate_fwd(a);
  if (s != FA_OK) return s;
  return fa::launch_simt(a);
}

fa_status fa_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int T, int d, float scale, int causal, fa_dtype dtype,
                       int num_splits, void* workspace, unsigned long long workspace_bytes,
                       void* stream) {
  fa::FwdArgs a{q, k, v, o, lse, B, Hq, Hkv, T, d, scale, causal, dtype,
                static_cast<cudaStream_t>(stream)};
  fa_status s = fa::validate_fwd(a);
  if (s != FA_OK) return s;
  if (num_splits < 1 || num_splits > fa::kMaxSplits) return FA_ERR_INVALID_ARG;
  if (dtype == FA_DTYPE_F32) return fa::launch_simt(a);
  if (num_splits == 1) return fa::launch_tc(a);
  if (workspace == nullptr) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 15u) return FA_ERR_MISALIGNED;
  const size_t need = fa::split_workspace_bytes(B, Hq, T, d, num_splits);
  if (workspace_bytes < need) return FA_ERR_WORKSPACE;
  const size_t e = 2;
  const size_t nq = static_cast<size_t>(B) * Hq * T * d * e;
  const size_t nkv = static_cast<size_t>(B) * Hkv * T * d * e;
  const size_t nl = static_cast<size_t>(B) * Hq * T * 4;
  if (fa::overlap(workspace, need, q, nq) || fa::overlap(workspace, need, k, nkv) ||
      fa::overlap(workspace, need, v, nkv) || fa::overlap(workspace, need, o, nq) ||
      fa::overlap(workspace, need, lse, nl))
    return FA_ERR_INVALID_ARG;
  return fa::launch_tc_split(a, num_splits, workspace, workspace_bytes);
}

}  // extern "C"

namespace fa {

// The backward entry points: checks, then the row preparation and the
// gradient kernels.  With lg_tokens >= 0 (local-global mask; the window is
// the local window on both sides) the key sets are built in the workspace
// after the rows' part.
static fa_status bwd_entry(const void* q, const void* k, const void* v, const void* o,
                           const float* lse, const void* d_o, void* dq, void* dk, void* dv, int B,
                           int Hq, int Hkv, int T, int d, float scale, int causal,
                           int window_left, int window_right, const int* lg_tokens,
                           int lg_num, fa_dtype dtype, void* workspace,
                           unsigned long long workspace_bytes, void* stream) {
  // the forward's checks cover q, k, v (as inputs), o and lse (as the
  // "outputs" that must not overlap them) and every size
  FwdArgs f{q, k, v, const_cast<void*>(o), const_cast<float*>(lse), B, Hq, Hkv, T, d, scale,
            causal, dtype, static_cast<cudaStream_t>(stream)};
  if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
  fa_status s = validate_fwd(f);
  if (s != FA_OK) return s;
  if (!d_o || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned16(d_o) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_MISALIGNED;
  const bool lg = lg_num >= 0;
  if (lg && lg_num > 0 && lg_tokens == nullptr) return FA_ERR_INVALID_ARG;
  if (lg && (reinterpret_cast<uintptr_t>(lg_tokens) & 3u)) return FA_ERR_MISALIGNED;
  if (workspace == nullptr) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 15u) return FA_ERR_MISALIGNED;
  const size_t rows_bytes = bwd_workspace_bytes(B, Hq, T);
  const size_t need = rows_bytes + (lg ? lg_workspace_bytes(T) : 0);
  if (workspace_bytes < need) return FA_ERR_WORKSPACE;
  const size_t e = dtype == FA_DTYPE_F32 ? 4 : 2;
  const size_t nq = static_cast<size_t>(B) * Hq * T * d * e;
  const size_t nkv = static_cast<size_t>(B) * Hkv * T * d * e;
  const size_t nl = static_cast<size_t>(B) * Hq * T * 4;
  const size_t ng = lg ? static_cast<size_t>(lg_num) * 4 : 0;
  // every written buffer (dq, dk, dv, workspace) against every other buffer
  const void* bufs[11] = {q, k, v, o, lse, d_o, lg_tokens, dq, dk, dv, workspace};
  const size_t lens[11] = {nq, nkv, nkv, nq, nl, nq, ng, nq, nkv, nkv, need};
  for (int w = 7; w < 11; ++w)
    for (int x = 0; x < 11; ++x)
      if (x != w && lens[x] > 0 && overlap(bufs[w], lens[w], bufs[x], lens[x]))
        return FA_ERR_INVALID_ARG;
  BwdArgs a{q, k, v, o, lse, d_o, dq, dk, dv, B, Hq, Hkv, T, d, scale, causal,
            window_left, window_right, dtype, static_cast<float*>(workspace),
            static_cast<float*>(workspace) + static_cast<size_t>(B) * Hq * bwd_rows_padded(T),
            static_cast<cudaStream_t>(stream)};
  if (lg) {
    LgSets g;
    s = lg_prep(T, lg_tokens, lg_num, static_cast<uint8_t*>(workspace) + rows_bytes, a.stream,
                &g);
    if (s != FA_OK) return s;
    a.local_global = true;
    a.lg_bits = g.bits;
    a.lg_list = g.list;
    a.lg_count = g.count;
  }
  s = launch_bwd_prep(a);
  if (s != FA_OK) return s;
  return bwd_tc_supported(a) ? launch_bwd_tc(a) : launch_bwd_simt(a);
}

}  // namespace fa

extern "C" {

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* d_o, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int T,
                 int d, float scale, int causal, int window_left, int window_right,
                 fa_dtype dtype, void* workspace, unsigned long long workspace_bytes,
                 void* stream) {
  return fa::bwd_entry(q, k, v, o, lse, d_o, dq, dk, dv, B, Hq, Hkv, T, d, scale, causal,
                       window_left, window_right, nullptr, -1, dtype, workspace,
                       workspace_bytes, stream);
}

fa_status fa_bwd_local_global(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* d_o, void* dq, void* dk, void* dv,
                              int B, int Hq, int Hkv, int T, int d, float scale, int causal,
                              int local_window, const int* global_tokens, int num_global,
                              fa_dtype dtype, void* workspace,
                              unsigned long long workspace_bytes, void* stream) {
  if (local_window < 0 || num_global < 0) return FA_ERR_INVALID_ARG;
  return fa::bwd_entry(q, k, v, o, lse, d_o, dq, dk, dv, B, Hq, Hkv, T, d, scale, causal,
                       local_window, local_window, global_tokens, num_global, dtype, workspace,
                       workspace_bytes, stream);
}

unsigned long long fa_bwd_local_global_workspace_size(int B, int Hq, int T) {
  if (B <= 0 || Hq <= 0 || T <= 0) return 0;
  return fa::bwd_workspace_bytes(B, Hq, T) + fa::lg_workspace_bytes(T);
}

fa_status fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int Hq, int Hkv, int T, int d, float scale, int causal, fa_dtype dtype,
                      int chunks, void* workspace, unsigned long long workspace_bytes,
                      void* stream) {
  fa::FwdArgs a{q, k, v, o, lse, B, Hq, Hkv, T, d, scale, causal, dtype,
                static_cast<cudaStream_t>(stream)};
  fa_status s = fa::validate_fwd(a);
  if (s != FA_OK) return s;
  if (chunks < 1) return FA_ERR_INVALID_ARG;
  if (chunks > B) chunks = B;
  if (workspace == nullptr) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 15u) return FA_ERR_MISALIGNED;
  if (workspace_bytes < fa::host_workspace_bytes(B, Hq, Hkv, T, d, dtype, chunks))
    return FA_ERR_WORKSPACE;
  return fa::run_fwd_host(a, chunks, workspace);
}

fa_status fa_bwd_host(const void* q, const void* k, const void* v, const void* o, const float* lse,
                      const void* d_o, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                      int T, int d, float scale, int causal, int window_left, int window_right,
                      fa_dtype dtype, int chunks, void* workspace,
                      unsigned long long workspace_bytes, void* stream) {
  fa::FwdArgs f{q, k, v, const_cast<void*>(o), const_cast<float*>(lse), B, Hq, Hkv, T, d, scale,
                causal, dtype, static_cast<cudaStream_t>(stream)};
  if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
  fa_status s = fa::validate_fwd(f);
  if (s != FA_OK) return s;
  if (!d_o || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!fa::aligned16(d_o) || !fa::aligned16(dq) || !fa::aligned16(dk) || !fa::aligned16(dv))
    return FA_ERR_MISALIGNED;
  if (chunks < 1) return FA_ERR_INVALID_ARG;
  if (chunks > B) chunks = B;
  if (workspace == nullptr) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 15u) return FA_ERR_MISALIGNED;
  if (workspace_bytes < fa::bwd_host_workspace_bytes(B, Hq, Hkv, T, d, dtype, chunks))
    return FA_ERR_WORKSPACE;
  const size_t e = dtype == FA_DTYPE_F32 ? 4 : 2;
  const size_t nq = static_cast<size_t>(B) * Hq * T * d * e;
  const size_t nkv = static_cast<size_t>(B) * Hkv * T * d * e;
  const size_t nl = static_cast<size_t>(B) * Hq * T * 4;
  // the host gradients against every host buffer
  const void* bufs[9] = {q, k, v, o, lse, d_o, dq, dk, dv};
  const size_t lens[9] = {nq, nkv, nkv, nq, nl, nq, nq, nkv, nkv};
  for (int w = 6; w < 9; ++w)
    for (int x = 0; x < 9; ++x)
      if (x != w && fa::overlap(bufs[w], lens[w], bufs[x], lens[x])) return FA_ERR_INVALID_ARG;
  fa::BwdArgs a{q, k, v, o, lse, d_o, dq, dk, dv, B, Hq, Hkv, T, d, scale, causal,
                window_left, window_right, dtype, nullptr, nullptr,
                static_cast<cudaStream_t>(stream)};
  return fa::run_bwd_host(a, chunks, workspace);
}

unsigned long long fa_bwd_host_workspace_size(int B, int Hq, int Hkv, int T, int d,
                                              fa_dtype dtype, int chunks) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || d <= 0 || chunks < 1) return 0;
  if (dtype != FA_DTYPE_F32 && dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F16) return 0;
  return fa::bwd_host_workspace_bytes(B, Hq, Hkv, T, d, dtype, chunks > B ? B : chunks);
}

unsigned long long fa_fwd_host_workspace_size(int B, int Hq, int Hkv, int T, int d,
                                              fa_dtype dtype, int chunks) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || d <= 0 || chunks < 1) return 0;
  if (dtype != FA_DTYPE_F32 && dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F16) return 0;
  return fa::host_workspace_bytes(B, Hq, Hkv, T, d, dtype, chunks > B ? B : chunks);
}

unsigned long long fa_bwd_workspace_size(int B, int Hq, int T) {
  if (B <= 0 || Hq <= 0 || T <= 0) return 0;
  return fa::bwd_workspace_bytes(B, Hq, T);
}

unsigned long long fa_fwd_split_workspace_size(int B, int Hq, int T, int d, int num_splits) {
  if (B <= 0 || Hq <= 0 || T <= 0 || d <= 0 || num_splits < 1 || num_splits > fa::kMaxSplits)
    return 0;
  return fa::split_workspace_bytes(B, Hq, T, d, num_splits);
}

int fa_fwd_split_heuristic(int B, int Hq, int Hkv, int T, int d, int causal) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || d <= 0) return 1;
  return fa::split_heuristic(B, Hq, T, causal);
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported head dimension or dtype";
    case FA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "kernel barrier wait timed out";
    case FA_ERR_WORKSPACE: return "scratch workspace missing or too small";
    default: return "unknown status";
  }
}

int fa_version(void) { return 10000; }

int fa_last_cuda_error(void) { return fa::t_last_cuda_error; }

fa_status fa_debug_sync_check(void* stream) {
  unsigned int word = 0;
  fa_status s = fa::read_and_clear_device_error(static_cast<cudaStream_t>(stream), &word);
  if (s != FA_OK) return s;
  return word ? FA_ERR_TIMEOUT : FA_OK;
}

}  // extern "C"
