// fa_internal.h -- declarations shared by the translation units of libfa.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/fa.h"

namespace fa {

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, Hq, Hkv, T, d;
  float scale;
  int causal;
  fa_dtype dtype;
  cudaStream_t stream;
  // band mask: keep key j for query i iff i - window_left <= j <= i + window_right
  // (-1 = unbounded side); combined with `causal` by intersection
  int window_left = -1;
  int window_right = -1;
  // local-global mask (window_left = window_right = the local window): keys
  // flagged in lg_bits are kept for every row as well, then causal applies.
  // lg_bits: one bit per key, 4 words per 128-key tile; lg_list: the sorted
  // tiles holding a flagged key, lg_count of them (written by launch_lg_prep)
  bool local_global = false;
  const uint32_t* lg_bits = nullptr;
  const int* lg_list = nullptr;
  const int* lg_count = nullptr;
  // packed global keys (16-bit tensor-core path, launch_lg_pack): the sorted
  // distinct global tokens lg_tokens[0, *lg_ntok) and their K and V rows
  // gathered into lg_kg, lg_vg, [B*Hkv][lg_rows][d] (lg_rows: a multiple of
  // 128; rows past the token count are zero)
  bool lg_packed = false;
  const int* lg_tokens = nullptr;
  const int* lg_ntok = nullptr;
  const void* lg_kg = nullptr;
  const void* lg_vg = nullptr;
  int lg_rows = 0;
};

// Workspace of the local-global mask for T keys: the key bitmask (16 bytes
// per 128-key tile), the list of tiles holding a global key (4 bytes per
// tile) and the list's length.
size_t lg_workspace_bytes(int T);
// Builds the bitmask and the tile list from `num_global` key indices (any
// order; repeats and entries outside [0, T) select nothing more) into
// `workspace` (lg_workspace_bytes(T) bytes) on `stream`.
struct LgSets {
  const uint32_t* bits;
  const int* list;
  const int* count;
};
fa_status lg_prep(int T, const int* global_tokens, int num_global, void* workspace,
                  cudaStream_t stream, LgSets* out);
// The same for a forward call: points a.lg_* at the sets.
fa_status launch_lg_prep(FwdArgs& a, const int* global_tokens, int num_global, void* workspace);

// Workspace of the packed global keys on top of lg_workspace_bytes(T): the
// sorted distinct tokens (lg_pack_rows(num_global) ints), their count, and the
// K and V rows gathered per (b, KV head): 2 * B * Hkv * rows * d * elem bytes,
// rows = num_global rounded up to a multiple of 128.
int lg_pack_rows(int num_global);
size_t lg_pack_workspace_bytes(int B, int Hkv, int d, size_t elem, int num_global);
// After launch_lg_prep: compacts the bitmask into the sorted token list and
// gathers the K, V rows into `pack_ws` (lg_pack_workspace_bytes bytes, 16-byte
// aligned); sets a.lg_packed and the a.lg_* pointers of the packed keys.
fa_status launch_lg_pack(FwdArgs& a, int num_global, void* pack_ws);

// The band the kernels apply: the window intersected with causal (j <= i).
// A side of T - 1 or more reaches every key, so it becomes unbounded (-1):
// the kernels' band arithmetic then stays within a few T (T < 2^30).
inline void band_of(int window_left, int window_right, int causal, int T, int& wl, int& wr) {
  wl = window_left >= T - 1 ? -1 : window_left;
  wr = window_right >= T - 1 ? -1 : window_right;
  if (causal) wr = 0;  // min(wr, 0) for wr >= 0, and 0 for an unbounded wr
}
inline void effective_window(const FwdArgs& a, int& wl, int& wr) {
  band_of(a.window_left, a.window_right, a.causal, a.T, wl, wr);
}

// One-time setup per kernel and device (kernel attributes such as the dynamic
// shared-memory limit are per device): the current device's slot in a
// per-kernel table, or nullptr for a device index past the table (the caller
// then repeats the setup on every call: correct, only slower).
inline bool* device_flag(bool (&flags)[64]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  return &flags[dev];
}

// Host-side argument checks shared by every entry point (no CUDA calls).
fa_status validate_fwd(const FwdArgs& a);
bool overlap(const void* a, size_t na, const void* b, size_t nb);

// Records a CUDA error for fa_last_cuda_error() and maps it to a status.
fa_status cuda_status(cudaError_t e);
fa_status cu_status(CUresult r);

// 3-D tensor map over a contiguous [BH][T][d] tensor of 16-bit elements
// (fp16 when f16, else bf16) with boxes of box_x columns x box_rows rows x 1
// and the given swizzle (CUtensorMapSwizzle).
CUresult make_tmap_16bit(CUtensorMap* map, const void* base, int d, int T, long long BH,
                         int box_x, int swizzle, bool f16, int box_rows = 128);
inline CUresult make_tmap_bf16(CUtensorMap* map, const void* base, int d, int T, long long BH,
                               int box_x, int swizzle) {
  return make_tmap_16bit(map, base, d, T, BH, box_x, swizzle, false);
}

// Kernel launchers (enqueue only; arguments already validated).
fa_status launch_tc(const FwdArgs& a);    // bf16 / fp16, tcgen05
// the same with the KV range of every row block split S ways: partial
// results go to `workspace` (split_workspace_bytes(...) bytes), a second
// kernel merges them into o and lse
fa_status launch_tc_split(const FwdArgs& a, int S, void* workspace, size_t workspace_bytes);
size_t split_workspace_bytes(int B, int Hq, int T, int d, int S);
int split_heuristic(int B, int Hq, int T, int causal);
constexpr int kMaxSplits = 64;
fa_status launch_simt(const FwdArgs& a);  // fp32, bf16 or fp16, CUDA cores

// ------------------------------------------------------------- backward
struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const float* lse;
  const void* d_o;
  void* dq;
  void* dk;
  void* dv;
  int B, Hq, Hkv, T, d;
  float scale;
  int causal;
  int window_left, window_right;
  fa_dtype dtype;
  float* ws_delta;  // [B*Hq][Tp] D_i = sum_c dO[i][c] O[i][c] (0 on padded rows)
  float* ws_lse2;   // [B*Hq][Tp] lse_i * log2(e) (+inf on padded rows)
  cudaStream_t stream;
  // local-global mask (window_left = window_right = the local window), as in
  // FwdArgs
  bool local_global = false;
  const uint32_t* lg_bits = nullptr;
  const int* lg_list = nullptr;
  const int* lg_count = nullptr;
};

// Query rows per head in the workspace: T rounded up to a multiple of 128.
inline int bwd_rows_padded(int T) { return (T + 127) / 128 * 128; }
size_t bwd_workspace_bytes(int B, int Hq, int T);

inline void effective_window(const BwdArgs& a, int& wl, int& wr) {
  band_of(a.window_left, a.window_right, a.causal, a.T, wl, wr);
}

// D and lse * log2(e) into the workspace (CUDA cores; any dtype)
fa_status launch_bwd_prep(const BwdArgs& a);
// dQ, dK, dV with fp32 FFMA (any dtype and d)
fa_status launch_bwd_simt(const BwdArgs& a);
// dQ, dK, dV on the tensor cores (bf16 / fp16, d in {64, 128})
fa_status launch_bwd_tc(const BwdArgs& a);
bool bwd_tc_supported(const BwdArgs& a);
fa_status bwd_read_and_clear_error(unsigned int* word);

// ------------------------------------------------------------- host buffers
// Device workspace of fa_fwd_host: two chunk slots of Q, K, V, O and LSE.
size_t host_workspace_bytes(int B, int Hq, int Hkv, int T, int d, fa_dtype dtype, int chunks);
// Forward from host q, k, v to host o, lse (a.* hold host pointers), in
// `chunks` batch chunks pipelined over two internal streams.
fa_status run_fwd_host(const FwdArgs& a, int chunks, void* workspace);
// Device workspace of fa_bwd_host, and the backward from host buffers (a.*
// hold host pointers; a.ws_* are unused: each chunk slot holds its own rows)
size_t bwd_host_workspace_bytes(int B, int Hq, int Hkv, int T, int d, fa_dtype dtype,
                                int chunks);
fa_status run_bwd_host(const BwdArgs& a, int chunks, void* workspace);

// Device error word shared by the kernels (read-and-clear, synchronous).
fa_status read_and_clear_device_error(cudaStream_t stream, unsigned int* word);

}  // namespace fa
