// fa_mask.cu -- the key sets of the local-global mask.
//
// The yelogs.com Flash Attention2/Triton tutorial, section "1. 稀疏注意力支持",
// defines the local-global mask as |i - j| <= local_window OR the key j is one
// of the listed global tokens (torch.isin over the key index).  The attention
// kernels need that list in two forms, built here on the device:
//   * a bitmask with one bit per key (4 words per 128-key tile), which the
//     masking step reads for the tiles it has to mask;
//   * the sorted list of 128-key tiles holding at least one global key, which
//     decides the KV tiles a query tile visits besides those of its band;
//   * for the 16-bit tensor-core forward, when the caller's workspace has
//     room: the sorted list of the distinct global tokens and their K and V
//     rows gathered into packed 128-row tiles, so that a query tile visits
//     ceil(#tokens / 128) packed tiles instead of one tile per global key.
// Entries outside [0, T) and repeats select nothing more (isin semantics).
#include <algorithm>

#include "fa_internal.h"

namespace fa {

namespace {

__global__ void __launch_bounds__(256)
    lg_scatter_kernel(const int* __restrict__ tokens, int n, uint32_t* __restrict__ bits, int T) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int t = tokens[i];
    if (t >= 0 && t < T) atomicOr(&bits[t >> 5], 1u << (t & 31));
  }
}

// One CTA of 1024 threads: compacts the tiles with a set bit, in order.
__global__ void __launch_bounds__(1024)
    lg_tiles_kernel(const uint32_t* __restrict__ bits, int n_tiles, int* __restrict__ list,
                    int* __restrict__ count) {
  __shared__ int warp_sum[32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < n_tiles; base += 1024) {
    const int t = base + tid;
    bool flag = false;
    if (t < n_tiles) {
      const uint4 w = reinterpret_cast<const uint4*>(bits)[t];
      flag = (w.x | w.y | w.z | w.w) != 0u;
    }
    const unsigned m = __ballot_sync(0xffffffffu, flag);
    if (lane == 0) warp_sum[warp] = __popc(m);
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < 32; ++w) {
      const int c = warp_sum[w];
      if (w < warp) before += c;
      total += c;
    }
    const int pos = carry + before + __popc(m & ((1u << lane) - 1u));
    if (flag) list[pos] = t;
    __syncthreads();  // every thread has read carry and warp_sum
    if (tid == 0) carry += total;
    __syncthreads();
  }
  if (tid == 0) *count = carry;
}

// One CTA of 1024 threads: the positions of the set bits of bits[0, n_words)
// in increasing order (a block-wide scan of the per-word bit counts).
__global__ void __launch_bounds__(1024)
    lg_tokens_kernel(const uint32_t* __restrict__ bits, int n_words, int* __restrict__ tokens,
                     int* __restrict__ count) {
  __shared__ int warp_sum[32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < n_words; base += 1024) {
    const int w = base + tid;
    uint32_t word = w < n_words ? bits[w] : 0u;
    const int c = __popc(word);
    int incl = c;  // inclusive scan of the counts within the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    int before = 0, total = 0;
    for (int x = 0; x < 32; ++x) {
      const int v = warp_sum[x];
      if (x < warp) before += v;
      total += v;
    }
    int pos = carry + before + incl - c;
    while (word != 0u) {
      const int b = __ffs(static_cast<int>(word)) - 1;
      tokens[pos++] = w * 32 + b;
      word &= word - 1u;
    }
    __syncthreads();  // every thread has read carry and warp_sum
    if (tid == 0) carry += total;
    __syncthreads();
  }
  if (tid == 0) *count = carry;
}

// Packed rows: row p of (b, KV head) z is row tokens[p] of K (and V) for
// p < *count, zero past it.  One thread per 16-byte piece of a row.
__global__ void __launch_bounds__(256)
    lg_gather_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                     uint4* __restrict__ kg, uint4* __restrict__ vg,
                     const int* __restrict__ tokens, const int* __restrict__ count, int T,
                     int rows, int pieces, long long n) {
  const int ntok = *count;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / pieces;  // packed row over all (b, KV head)
    const int c = static_cast<int>(i - r * pieces);
    const long long z = r / rows;
    const int p = static_cast<int>(r - z * rows);
    uint4 kx = make_uint4(0u, 0u, 0u, 0u), vx = kx;
    if (p < ntok) {
      const long long src = (z * T + tokens[p]) * pieces + c;
      kx = k[src];
      vx = v[src];
    }
    kg[i] = kx;
    vg[i] = vx;
  }
}

}  // namespace

size_t lg_workspace_bytes(int T) {
  const size_t tiles = (static_cast<size_t>(T) + 127) / 128;
  return (tiles * 16 + tiles * 4 + 16 + 15) / 16 * 16;
}

fa_status lg_prep(int T, const int* global_tokens, int num_global, void* workspace,
                  cudaStream_t stream, LgSets* out) {
  const int n_tiles = (T + 127) / 128;
  uint32_t* bits = static_cast<uint32_t*>(workspace);
  int* list = reinterpret_cast<int*>(bits + static_cast<size_t>(n_tiles) * 4);
  int* count = list + n_tiles;
  cudaError_t e = cudaMemsetAsync(bits, 0, static_cast<size_t>(n_tiles) * 16, stream);
  if (e != cudaSuccess) return cuda_status(e);
  if (num_global > 0) {
    const int blocks = static_cast<int>(std::min<long long>((num_global + 255) / 256, 1024));
    lg_scatter_kernel<<<blocks, 256, 0, stream>>>(global_tokens, num_global, bits, T);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e);
  }
  lg_tiles_kernel<<<1, 1024, 0, stream>>>(bits, n_tiles, list, count);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_status(e);
  out->bits = bits;
  out->list = list;
  out->count = count;
  return FA_OK;
}

int lg_pack_rows(int num_global) {
  return static_cast<int>(std::max<long long>(128, (static_cast<long long>(num_global) + 127) / 128 * 128));
}

size_t lg_pack_workspace_bytes(int B, int Hkv, int d, size_t elem, int num_global) {
  const size_t rows = static_cast<size_t>(lg_pack_rows(num_global));
  return rows * 4 + 16 + 2 * static_cast<size_t>(B) * Hkv * rows * d * elem;
}

fa_status launch_lg_pack(FwdArgs& a, int num_global, void* pack_ws) {
  const int rows = lg_pack_rows(num_global);
  int* tokens = static_cast<int*>(pack_ws);
  int* ntok = tokens + rows;
  uint8_t* kg = reinterpret_cast<uint8_t*>(ntok) + 16;
  const size_t row_bytes = static_cast<size_t>(a.d) * 2;  // 16-bit elements
  const size_t plane = static_cast<size_t>(a.B) * a.Hkv * rows * row_bytes;
  uint8_t* vg = kg + plane;
  const int n_words = (a.T + 127) / 128 * 4;
  lg_tokens_kernel<<<1, 1024, 0, a.stream>>>(a.lg_bits, n_words, tokens, ntok);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_status(e);
  const int pieces = static_cast<int>(row_bytes / 16);
  const long long n = static_cast<long long>(plane / 16);
  const int blocks = static_cast<int>(std::min<long long>((n + 255) / 256, 4096));
  lg_gather_kernel<<<blocks, 256, 0, a.stream>>>(
      static_cast<const uint4*>(a.k), static_cast<const uint4*>(a.v), reinterpret_cast<uint4*>(kg),
      reinterpret_cast<uint4*>(vg), tokens, ntok, a.T, rows, pieces, n);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_status(e);
  a.lg_packed = true;
  a.lg_tokens = tokens;
  a.lg_ntok = ntok;
  a.lg_kg = kg;
  a.lg_vg = vg;
  a.lg_rows = rows;
  return FA_OK;
}

fa_status launch_lg_prep(FwdArgs& a, const int* global_tokens, int num_global, void* workspace) {
  LgSets g;
  const fa_status s = lg_prep(a.T, global_tokens, num_global, workspace, a.stream, &g);
  if (s != FA_OK) return s;
  a.local_global = true;
  a.lg_bits = g.bits;
  a.lg_list = g.list;
  a.lg_count = g.count;
  return FA_OK;
}

}  // namespace fa
