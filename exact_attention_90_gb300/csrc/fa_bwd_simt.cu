// fa_bwd_simt.cu -- attention backward with true-fp32 FFMA on the CUDA cores,
// and the row preparation that every backward path uses.
//
// The backward recomputes the forward's probabilities instead of storing them
// ("Flash Attention Memory Optimization Explained", section "Key Mechanisms",
// item "Backward Checkpointing"): P = exp(S - lse) from the forward's per-row
// log-sum-exp, tile by tile.  With D_i = sum_c dO[i][c] O[i][c] (which equals
// sum_j P_ij dP_ij because O = P V):
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  dQ = scale dS K,
//   dK = scale dS^T Q  (dK, dV summed over the query heads sharing a KV head).
//
// Three kernels:
//   fa_bwd_prep_kernel      -- per query row: -D_i and -lse_i * log2(e) into
//                              the workspace (padded rows: 0 and -inf, so that
//                              a padded query gets P = 0);
//   fa_bwd_dq_simt_kernel   -- one CTA per 64 query rows: loops over the KV
//                              blocks of the band, accumulates dQ in registers;
//   fa_bwd_dkdv_simt_kernel -- one CTA per 64 keys of a KV head: loops over the
//                              query heads of its group and their query blocks,
//                              accumulates dK and dV in registers.
// No gradient is accumulated across CTAs, so results are deterministic.
// Thread layout as in the forward CUDA-core kernel (fa_simt.cu): 128 threads
// as a 16 x 8 grid, thread (tx, ty) owns tile rows ty*8 .. ty*8+7, columns
// tx*4 .. tx*4+3 of the 64 x 64 score tile and d/16 output columns.
#include <cmath>

#include "fa_internal.h"
#include "simt_tiles.cuh"

namespace fa {

namespace {

using namespace simt;

constexpr float kLog2e = 1.4426950408889634f;

template <typename Tin>
__device__ __forceinline__ float to_f32(Tin x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }

// 2^x on the special-function unit (documented PTX instruction; relative
// error about 2^-22, far inside the fp32 gradient tolerance)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// sum over the elements of two 16-byte vectors of products a * b
template <typename Tin>
__device__ __forceinline__ float dot16(const uint4& a, const uint4& b) {
  constexpr int VEC = 16 / static_cast<int>(sizeof(Tin));
  const Tin* x = reinterpret_cast<const Tin*>(&a);
  const Tin* y = reinterpret_cast<const Tin*>(&b);
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc = fmaf(to_f32(x[e]), to_f32(y[e]), acc);
  return acc;
}

// -D_i = -sum_c dO[i][c] * O[i][c] and -lse_i * log2(e) per padded row.  Stored
// negated, so that the tensor-core kernels add them with paired fp32 adds and
// FMAs; padded rows get -D = 0 and -lse log2(e) = -inf (P = 0).  A row is read
// by d * sizeof(Tin) / 16 consecutive lanes (2 to 32, a power of two), one
// 16-byte load of O and of dO each, and reduced by shuffles within that group.
template <typename Tin>
__global__ void __launch_bounds__(256)
    fa_bwd_prep_kernel(const Tin* __restrict__ o, const Tin* __restrict__ d_o,
                       const float* __restrict__ lse, float* __restrict__ delta,
                       float* __restrict__ lse2, long long BH, int T, int Tp, int d) {
  constexpr int VEC = 16 / static_cast<int>(sizeof(Tin));
  const int L = d / VEC;  // lanes per row
  const long long gtid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = gtid / L;
  const int sub = static_cast<int>(gtid - row * L);
  const bool active = row < BH * Tp;
  long long bh = 0;
  int i = 0;
  float acc = 0.f;
  if (active) {
    bh = row / Tp;
    i = static_cast<int>(row - bh * Tp);
    if (i < T) {
      const size_t base = (static_cast<size_t>(bh) * T + i) * d + static_cast<size_t>(sub) * VEC;
      acc = dot16<Tin>(*reinterpret_cast<const uint4*>(o + base),
                       *reinterpret_cast<const uint4*>(d_o + base));
    }
  }
  // the row's lanes are an aligned group of L inside the warp (L divides 32)
  for (int off = L >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (active && sub == 0) {
    delta[row] = -acc;
    lse2[row] = i < T ? -(lse[static_cast<size_t>(bh) * T + i] * kLog2e) : -INFINITY;
  }
}

// keep key j for query i: inside [0, T) and the band i - wl <= j <= i + wr,
// or (local-global masks, lg_bits != nullptr) j is a global key, not after i
// when lg_causal
__device__ __forceinline__ bool band_keep(int i, int j, int T, int wl, int wr,
                                          const uint32_t* lg_bits = nullptr, int lg_causal = 0) {
  if (i >= T || j >= T) return false;
  if ((wr < 0 || j <= i + wr) && (wl < 0 || j >= i - wl)) return true;
  return lg_bits != nullptr && (!lg_causal || j <= i) &&
         ((__ldg(lg_bits + (j >> 5)) >> (j & 31)) & 1u) != 0u;
}

// any global key in the 64-key block kb0 .. kb0 + 63 (two bitmask words)
__device__ __forceinline__ bool block_has_global(const uint32_t* lg_bits, int kb0) {
  return (__ldg(lg_bits + (kb0 >> 5)) | __ldg(lg_bits + (kb0 >> 5) + 1)) != 0u;
}

// acc[8][OC] += A[rows ty*8.., 0..63] (stride PS) x B[0..63][cols] (stride BS)
template <int D, int BS>
__device__ __forceinline__ void simt_acc_product(float (&acc)[8][D / 16], const float* sA,
                                                 const float* sB, int tx, int ty) {
  constexpr int PS = SimtCfg<D>::PS, OC = SimtCfg<D>::OC;
  constexpr int GW = D >= 64 ? 4 : (D == 32 ? 2 : 1);
#pragma unroll 2
  for (int kk = 0; kk < 64; kk += 4) {
    float4 av[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) av[i] = *reinterpret_cast<const float4*>(sA + (ty * 8 + i) * PS + kk);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float bv[OC];
      const float* br = sB + (kk + u) * BS;
#pragma unroll
      for (int c = 0; c < OC; c += GW) {
        if constexpr (GW == 4) {
          const float4 t4 = *reinterpret_cast<const float4*>(br + ocol<D>(tx, c));
          bv[c] = t4.x; bv[c + 1] = t4.y; bv[c + 2] = t4.z; bv[c + 3] = t4.w;
        } else if constexpr (GW == 2) {
          const float2 t2 = *reinterpret_cast<const float2*>(br + ocol<D>(tx, c));
          bv[c] = t2.x; bv[c + 1] = t2.y;
        } else {
          bv[c] = br[ocol<D>(tx, c)];
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float a = u == 0 ? av[i].x : (u == 1 ? av[i].y : (u == 2 ? av[i].z : av[i].w));
#pragma unroll
        for (int c = 0; c < OC; ++c) acc[i][c] = fmaf(a, bv[c], acc[i][c]);
      }
    }
  }
}

// x[8][4] = A[rows ty*8..] . B[cols tx*4..] over D (both stride QS), and the
// same for a second pair (y = C . E): the two score-shaped products of a tile
template <int D>
__device__ __forceinline__ void simt_two_dots(float (&x)[8][4], float (&y)[8][4], const float* sA,
                                              const float* sB, const float* sC, const float* sE,
                                              int tx, int ty) {
  constexpr int QS = SimtCfg<D>::QS;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int c = 0; c < 4; ++c) x[i][c] = y[i][c] = 0.f;
#pragma unroll 2
  for (int kk = 0; kk < D; kk += 4) {
    float4 bv[4], ev[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      bv[c] = *reinterpret_cast<const float4*>(sB + (tx * 4 + c) * QS + kk);
      ev[c] = *reinterpret_cast<const float4*>(sE + (tx * 4 + c) * QS + kk);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 av = *reinterpret_cast<const float4*>(sA + (ty * 8 + i) * QS + kk);
      const float4 cv = *reinterpret_cast<const float4*>(sC + (ty * 8 + i) * QS + kk);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        x[i][c] = fmaf(av.x, bv[c].x, x[i][c]);
        x[i][c] = fmaf(av.y, bv[c].y, x[i][c]);
        x[i][c] = fmaf(av.z, bv[c].z, x[i][c]);
        x[i][c] = fmaf(av.w, bv[c].w, x[i][c]);
        y[i][c] = fmaf(cv.x, ev[c].x, y[i][c]);
        y[i][c] = fmaf(cv.y, ev[c].y, y[i][c]);
        y[i][c] = fmaf(cv.z, ev[c].z, y[i][c]);
        y[i][c] = fmaf(cv.w, ev[c].w, y[i][c]);
      }
    }
  }
}

template <typename Tin, int D>
__device__ __forceinline__ void store_rows(Tin* dst, const float (&acc)[8][D / 16], int r0, int T,
                                           int tx, int ty) {
  constexpr int OC = SimtCfg<D>::OC;
  constexpr int GW = D >= 64 ? 4 : (D == 32 ? 2 : 1);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = r0 + ty * 8 + i;
    if (row >= T) continue;
    Tin* r = dst + static_cast<size_t>(row) * D;
#pragma unroll
    for (int c = 0; c < OC; c += GW) {
      float y[4];
#pragma unroll
      for (int e = 0; e < GW; ++e) y[e] = acc[i][c + e];
      store_out(r + ocol<D>(tx, c), y, GW);
    }
  }
}

template <int D>
struct BwdSimtCfg {
  static constexpr int QS = SimtCfg<D>::QS, PS = SimtCfg<D>::PS;
  static constexpr int DQ_SMEM = (4 * 64 * QS + 64 * PS) * 4;
  static constexpr int DKDV_SMEM = (4 * 64 * QS + 2 * 64 * PS) * 4;
};

// dQ for 64 query rows of one (b, h): rows = queries, score columns = keys
template <typename Tin, int D>
__global__ void __launch_bounds__(128)
    fa_bwd_dq_simt_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                          const Tin* __restrict__ v, const Tin* __restrict__ d_o,
                          const float* __restrict__ delta, const float* __restrict__ lse2,
                          Tin* __restrict__ dq, int B, int Hq, int Hkv, int T, int Tp,
                          float scale, int wl, int wr, const uint32_t* __restrict__ lg_bits,
                          int lg_causal) {
  constexpr int QS = SimtCfg<D>::QS, PS = SimtCfg<D>::PS, OC = SimtCfg<D>::OC;
  extern __shared__ float4 smem4[];
  float* sQ = reinterpret_cast<float*>(smem4);
  float* sdO = sQ + 64 * QS;
  float* sK = sdO + 64 * QS;
  float* sV = sK + 64 * QS;
  float* sS = sV + 64 * QS;
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int BH = B * Hq;
  const int n_qt = (T + 63) / 64, n_kt = (T + 63) / 64;
  const int qt = n_qt - 1 - static_cast<int>(blockIdx.x / BH);
  const int bh = static_cast<int>(blockIdx.x % BH);
  const int b = bh / Hq, h = bh - b * Hq;
  const int hk = h / (Hq / Hkv);
  const int q0 = qt * 64;
  const size_t qoff = static_cast<size_t>(bh) * T * D;
  const size_t kvoff = static_cast<size_t>(b * Hkv + hk) * T * D;
  const float sl2 = scale * kLog2e;

  load_tile<D, QS>(sQ, q + qoff, q0, T);
  load_tile<D, QS>(sdO, d_o + qoff, q0, T);
  float Lr[8], Dr[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const size_t r = static_cast<size_t>(bh) * Tp + q0 + ty * 8 + i;  // < Tp: rows are padded
    Lr[i] = -lse2[r];  // the workspace holds -lse log2(e) and -D
    Dr[i] = -delta[r];
  }
  float acc[8][OC];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int c = 0; c < OC; ++c) acc[i][c] = 0.f;

  const int b_lo = wl < 0 ? 0 : max(0, q0 - wl) / 64;
  const int b_hi = wr < 0 ? n_kt : min(n_kt, min(T - 1, q0 + 63 + wr) / 64 + 1);
  // local-global: any block may hold global keys (up to the rows' last key
  // when causal); blocks with neither band keys nor global keys are skipped
  const int j_lo = lg_bits ? 0 : b_lo;
  const int j_hi = lg_bits ? (lg_causal ? min(n_kt, min(T - 1, q0 + 63) / 64 + 1) : n_kt) : b_hi;
  for (int j = j_lo; j < j_hi; ++j) {
    if (lg_bits && (j < b_lo || j >= b_hi) && !block_has_global(lg_bits, j * 64)) continue;
    __syncthreads();  // previous block's K, V and dS no longer in use
    load_tile<D, QS>(sK, k + kvoff, j * 64, T);
    load_tile<D, QS>(sV, v + kvoff, j * 64, T);
    __syncthreads();
    float s[8][4], dp[8][4];
    simt_two_dots<D>(s, dp, sQ, sK, sdO, sV, tx, ty);  // S = Q K^T, dP = dO V^T
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = q0 + ty * 8 + i;
      float ds[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int key = j * 64 + tx * 4 + c;
        const float p = band_keep(row, key, T, wl, wr, lg_bits, lg_causal)
                            ? ex2_approx(fmaf(s[i][c], sl2, -Lr[i]))
                            : 0.f;
        ds[c] = p * (dp[i][c] - Dr[i]) * scale;
      }
      *reinterpret_cast<float4*>(sS + (ty * 8 + i) * PS + tx * 4) =
          make_float4(ds[0], ds[1], ds[2], ds[3]);
    }
    __syncthreads();
    simt_acc_product<D, QS>(acc, sS, sK, tx, ty);  // dQ += dS K
  }
  store_rows<Tin, D>(dq + qoff, acc, q0, T, tx, ty);
}

// dK and dV for 64 keys of one (b, hk): rows = keys, score columns = queries
template <typename Tin, int D>
__global__ void __launch_bounds__(128)
    fa_bwd_dkdv_simt_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                            const Tin* __restrict__ v, const Tin* __restrict__ d_o,
                            const float* __restrict__ delta, const float* __restrict__ lse2,
                            Tin* __restrict__ dk, Tin* __restrict__ dv, int B, int Hq, int Hkv,
                            int T, int Tp, float scale, int wl, int wr,
                            const uint32_t* __restrict__ lg_bits, int lg_causal) {
  constexpr int QS = SimtCfg<D>::QS, PS = SimtCfg<D>::PS, OC = SimtCfg<D>::OC;
  extern __shared__ float4 smem4[];
  float* sK = reinterpret_cast<float*>(smem4);
  float* sV = sK + 64 * QS;
  float* sQ = sV + 64 * QS;
  float* sdO = sQ + 64 * QS;
  float* sP = sdO + 64 * QS;
  float* sS = sP + 64 * PS;
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int BHk = B * Hkv;
  const int n_t = (T + 63) / 64;
  const int kt = static_cast<int>(blockIdx.x / BHk);
  const int bhk = static_cast<int>(blockIdx.x % BHk);
  const int b = bhk / Hkv, hk = bhk - b * Hkv;
  const int group = Hq / Hkv;
  const int k0 = kt * 64;
  const size_t kvoff = static_cast<size_t>(bhk) * T * D;
  const float sl2 = scale * kLog2e;

  load_tile<D, QS>(sK, k + kvoff, k0, T);
  load_tile<D, QS>(sV, v + kvoff, k0, T);
  float adk[8][OC], adv[8][OC];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int c = 0; c < OC; ++c) adk[i][c] = adv[i][c] = 0.f;

  // query blocks holding queries [k0 - wr, k0 + 63 + wl] (the transposed band)
  int i_lo = wr < 0 ? 0 : max(0, k0 - wr) / 64;
  int i_hi = wl < 0 ? n_t : min(n_t, min(T - 1, k0 + 63 + wl) / 64 + 1);
  if (lg_bits != nullptr && block_has_global(lg_bits, k0)) {
    // a block with a global key is attended by every query (from the key on)
    i_lo = lg_causal ? min(i_lo, k0 / 64) : 0;
    i_hi = n_t;
  }
  for (int g = 0; g < group; ++g) {
    const int bh = b * Hq + hk * group + g;
    const size_t qoff = static_cast<size_t>(bh) * T * D;
    for (int it = i_lo; it < i_hi; ++it) {
      const int q0 = it * 64;
      __syncthreads();  // previous block's Q, dO, P and dS no longer in use
      load_tile<D, QS>(sQ, q + qoff, q0, T);
      load_tile<D, QS>(sdO, d_o + qoff, q0, T);
      __syncthreads();
      float s[8][4], dp[8][4];
      simt_two_dots<D>(s, dp, sK, sQ, sV, sdO, tx, ty);  // S^T = K Q^T, dP^T = V dO^T
      float Lc[4], Dc[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const size_t r = static_cast<size_t>(bh) * Tp + q0 + tx * 4 + c;
        Lc[c] = -lse2[r];  // the workspace holds -lse log2(e) and -D
        Dc[c] = -delta[r];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int key = k0 + ty * 8 + i;
        float p[4], ds[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int qi = q0 + tx * 4 + c;
          p[c] = band_keep(qi, key, T, wl, wr, lg_bits, lg_causal)
                     ? ex2_approx(fmaf(s[i][c], sl2, -Lc[c]))
                     : 0.f;
          ds[c] = p[c] * (dp[i][c] - Dc[c]) * scale;
        }
        *reinterpret_cast<float4*>(sP + (ty * 8 + i) * PS + tx * 4) =
            make_float4(p[0], p[1], p[2], p[3]);
        *reinterpret_cast<float4*>(sS + (ty * 8 + i) * PS + tx * 4) =
            make_float4(ds[0], ds[1], ds[2], ds[3]);
      }
      __syncthreads();
      simt_acc_product<D, QS>(adv, sP, sdO, tx, ty);  // dV += P^T dO
      simt_acc_product<D, QS>(adk, sS, sQ, tx, ty);   // dK += dS^T Q
    }
  }
  store_rows<Tin, D>(dk + kvoff, adk, k0, T, tx, ty);
  store_rows<Tin, D>(dv + kvoff, adv, k0, T, tx, ty);
}

template <typename Tin>
fa_status launch_prep_t(const BwdArgs& a) {
  const long long BH = static_cast<long long>(a.B) * a.Hq;
  const int Tp = bwd_rows_padded(a.T);
  const long long rows = BH * Tp;
  const long long lanes = rows * (a.d * static_cast<long long>(sizeof(Tin)) / 16);
  fa_bwd_prep_kernel<Tin><<<static_cast<unsigned>((lanes + 255) / 256), 256, 0, a.stream>>>(
      static_cast<const Tin*>(a.o), static_cast<const Tin*>(a.d_o), a.lse, a.ws_delta, a.ws_lse2,
      BH, a.T, Tp, a.d);
  return cuda_status(cudaGetLastError());
}

template <typename Tin, int D>
fa_status launch_bwd_simt_impl(const BwdArgs& a) {
  using C = BwdSimtCfg<D>;
  auto kq = fa_bwd_dq_simt_kernel<Tin, D>;
  auto kkv = fa_bwd_dkdv_simt_kernel<Tin, D>;
  static bool attr_done[64] = {};  // per instantiation and device; benign race
  bool* done = device_flag(attr_done);
  if (done == nullptr || !*done) {
    cudaError_t e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, C::DQ_SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, C::DKDV_SMEM);
    if (e != cudaSuccess) return cuda_status(e);
    if (done != nullptr) *done = true;
  }
  int wl, wr;
  effective_window(a, wl, wr);
  const int Tp = bwd_rows_padded(a.T);
  const int n_t = (a.T + 63) / 64;
  const long long gq = static_cast<long long>(a.B) * a.Hq * n_t;
  const long long gkv = static_cast<long long>(a.B) * a.Hkv * n_t;
  kkv<<<static_cast<unsigned>(gkv), 128, C::DKDV_SMEM, a.stream>>>(
      static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v),
      static_cast<const Tin*>(a.d_o), a.ws_delta, a.ws_lse2, static_cast<Tin*>(a.dk),
      static_cast<Tin*>(a.dv), a.B, a.Hq, a.Hkv, a.T, Tp, a.scale, wl, wr,
      a.local_global ? a.lg_bits : nullptr, a.causal);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_status(e);
  kq<<<static_cast<unsigned>(gq), 128, C::DQ_SMEM, a.stream>>>(
      static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v),
      static_cast<const Tin*>(a.d_o), a.ws_delta, a.ws_lse2, static_cast<Tin*>(a.dq), a.B, a.Hq,
      a.Hkv, a.T, Tp, a.scale, wl, wr, a.local_global ? a.lg_bits : nullptr, a.causal);
  return cuda_status(cudaGetLastError());
}

template <typename Tin>
fa_status launch_bwd_simt_t(const BwdArgs& a) {
  switch (a.d) {
    case 16: return launch_bwd_simt_impl<Tin, 16>(a);
    case 32: return launch_bwd_simt_impl<Tin, 32>(a);
    case 64: return launch_bwd_simt_impl<Tin, 64>(a);
    case 128: return launch_bwd_simt_impl<Tin, 128>(a);
    default: return FA_ERR_UNSUPPORTED;
  }
}

}  // namespace

size_t bwd_workspace_bytes(int B, int Hq, int T) {
  return static_cast<size_t>(2) * B * Hq * bwd_rows_padded(T) * sizeof(float);
}

fa_status launch_bwd_prep(const BwdArgs& a) {
  if (a.dtype == FA_DTYPE_F32) return launch_prep_t<float>(a);
  if (a.dtype == FA_DTYPE_BF16) return launch_prep_t<__nv_bfloat16>(a);
  if (a.dtype == FA_DTYPE_F16) return launch_prep_t<__half>(a);
  return FA_ERR_UNSUPPORTED;
}

fa_status launch_bwd_simt(const BwdArgs& a) {
  if (a.dtype == FA_DTYPE_F32) return launch_bwd_simt_t<float>(a);
  if (a.dtype == FA_DTYPE_BF16) return launch_bwd_simt_t<__nv_bfloat16>(a);
  if (a.dtype == FA_DTYPE_F16) return launch_bwd_simt_t<__half>(a);
  return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
