// fa_mask.cu -- the key sets of the local-global mask.
//
// The yelogs.com Flash Attention2/Triton tutorial, section "1. 稀疏注意力支持",
// defines the local-global mask as |i - j| <= local_window OR the key j is one
// of the listed global tokens (torch.isin over the key index).  The attention
// kernels need that list in two forms, built here on the device:
//   * a bitmask with one bit per key (4 words per 128-key tile), which the
//     masking step reads for the tiles it has to mask;
//   * the sorted list of 128-key tiles holding at least one global key, which
//     decides the KV tiles a query tile visits besides those of its band.
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
