// simt_tiles.cuh -- shared-memory tile helpers of the fp32 CUDA-core kernels
// (forward in fa_simt.cu, backward in fa_bwd_simt.cu): row tiles of a [T][D]
// matrix converted to fp32 in padded shared-memory rows, and
// vectorised stores of fp32 results in the output element type.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

namespace fa {
namespace simt {

constexpr int BQ = 64;
constexpr int BK = 64;

template <int D>
struct SimtCfg {
  static constexpr int QS = D + 4;  // padded row stride (floats) of Q and K
  static constexpr int PS = BK + 4; // padded row stride of P
  static constexpr int OC = D / 16; // output columns per thread
  static constexpr int SMEM_FLOATS = BQ * QS + BK * QS + BK * D + BQ * PS;
  static constexpr int SMEM_BYTES = SMEM_FLOATS * 4;
};

// Output column of a thread's c-th accumulator.
template <int D>
__device__ __forceinline__ int ocol(int tx, int c) {
  if constexpr (D >= 64) return tx * 4 + 64 * (c / 4) + (c % 4);
  else if constexpr (D == 32) return tx * 2 + c;
  else return tx;
}

// rows [r0, r0+ROWS) of a [T][D] matrix into smem (row stride LS floats),
// by the NT threads of the CTA; rows at or past T become zero
template <int D, int LS, int ROWS = 64, int NT = 128>
__device__ __forceinline__ void load_tile(float* dst, const float* src, int r0, int T) {
  constexpr int V = D / 4;  // float4 per row
#pragma unroll 4
  for (int idx = threadIdx.x; idx < ROWS * V; idx += NT) {
    const int r = idx / V, c4 = idx % V;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r0 + r < T) x = __ldg(reinterpret_cast<const float4*>(src + static_cast<size_t>(r0 + r) * D) + c4);
    *reinterpret_cast<float4*>(dst + r * LS + 4 * c4) = x;
  }
}

template <int D, int LS, int ROWS = 64, int NT = 128>
__device__ __forceinline__ void load_tile(float* dst, const __nv_bfloat16* src, int r0, int T) {
  constexpr int V = D / 8;  // 16-byte vectors of 8 bf16 per row
#pragma unroll 4
  for (int idx = threadIdx.x; idx < ROWS * V; idx += NT) {
    const int r = idx / V, c8 = idx % V;
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (r0 + r < T) x = __ldg(reinterpret_cast<const uint4*>(src + static_cast<size_t>(r0 + r) * D) + c8);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    float f[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[2 * e] = __uint_as_float(w[e] << 16);
      f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
    float* d = dst + r * LS + 8 * c8;
    *reinterpret_cast<float4*>(d) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4*>(d + 4) = make_float4(f[4], f[5], f[6], f[7]);
  }
}

template <int D, int LS, int ROWS = 64, int NT = 128>
__device__ __forceinline__ void load_tile(float* dst, const __half* src, int r0, int T) {
  constexpr int V = D / 8;  // 16-byte vectors of 8 fp16 per row
#pragma unroll 4
  for (int idx = threadIdx.x; idx < ROWS * V; idx += NT) {
    const int r = idx / V, c8 = idx % V;
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (r0 + r < T) x = __ldg(reinterpret_cast<const uint4*>(src + static_cast<size_t>(r0 + r) * D) + c8);
    const __half2* h = reinterpret_cast<const __half2*>(&x);
    float* d = dst + r * LS + 8 * c8;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(h[e]);
      d[2 * e] = f.x;
      d[2 * e + 1] = f.y;
    }
  }
}

__device__ __forceinline__ void store_out(__half* dst, const float* x, int n) {
  if (n == 4) {
    __half2 a = __floats2half2_rn(x[0], x[1]);
    __half2 b = __floats2half2_rn(x[2], x[3]);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(dst) = u;
  } else if (n == 2) {
    *reinterpret_cast<__half2*>(dst) = __floats2half2_rn(x[0], x[1]);
  } else {
    dst[0] = __float2half_rn(x[0]);
  }
}

__device__ __forceinline__ void store_out(float* dst, const float* x, int n) {
  if (n == 4) *reinterpret_cast<float4*>(dst) = make_float4(x[0], x[1], x[2], x[3]);
  else if (n == 2) *reinterpret_cast<float2*>(dst) = make_float2(x[0], x[1]);
  else dst[0] = x[0];
}

__device__ __forceinline__ void store_out(__nv_bfloat16* dst, const float* x, int n) {
  if (n == 4) {
    __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]);
    __nv_bfloat162 b = __floats2bfloat162_rn(x[2], x[3]);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(dst) = u;
  } else if (n == 2) {
    *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(x[0], x[1]);
  } else {
    dst[0] = __float2bfloat16_rn(x[0]);
  }
}

}  // namespace simt
}  // namespace fa
