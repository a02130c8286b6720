// fa_simt.cu -- true-fp32 exact attention forward on the CUDA cores.
//
// The same computation as the tensor-core kernel (see fa_tc.cu): the tiled
// forward with online softmax of the yelogs.com Flash Attention2/Triton
// tutorial, section "核心 Kernel 實現" -- Q block kept on chip, K/V blocks
// streamed, running max m, normaliser l and output accumulator in fp32, the
// accumulator rescaled by exp(m_old - m_new) per block (section "Softmax 的在線
// 計算"), O / l and L = m + log l at the end -- with every product done by FFMA
// in fp32.  fp32 inputs need this path: a TF32 tensor-core product would not
// keep O within 1e-4 of the exact result.  It also accepts bf16 and fp16 inputs
// (fp32 arithmetic), which the tests use as a cross-check of the tensor-core
// kernel.
//
// CTA = 2 FQ threads = a 16 x (FQ / 8) grid (tx, ty) over an FQ-query x
// 64-key block (FQ = 64 or 128): thread (tx, ty) owns query rows ty*8 ..
// ty*8+7, score columns tx*4 .. tx*4+3 and d/16 output columns; row maxima
// and sums combine the 16 threads of a row with warp shuffles.  Tiles live in
// shared memory with padded rows so the 16-byte loads of a quarter-warp hit
// distinct banks.  FQ = 128 gives eight warps per SM at d = 128 (the shared
// memory allows one CTA there) and halves the K/V loads per flop; the host
// takes it for d >= 64 when the grid still covers every SM.
//
// fp32 inputs outside local-global masks take the pipelined form (ASYNC):
// K and V blocks arrive by cp.async, K double-buffered, so that the next K
// loads during this block's S, softmax and P.V and the next V during the
// next block's S.  The softmax works in log2 units with ex2.approx (scores
// times scale * log2(e), L = (m + log2 l) ln 2), as the tensor-core kernel
// does; the max rounding of m cancels between l and L in the same way.
#include <cmath>
#include <type_traits>

#include "fa_internal.h"
#include "simt_tiles.cuh"

namespace fa {

namespace {

using namespace simt;

// Band mask: keep key j for query i iff i - wl <= j <= i + wr (wl or wr < 0:
// unbounded side); no mask is (-1, -1), causal attention (-1, 0).  With
// lg_bits (local-global mask: one bit per key) a flagged key is kept as well,
// up to the row itself when lg_causal.
// FQ query rows per CTA, 2 FQ threads (16 per 8 rows x 64 keys)
template <int D, int FQ, bool ASYNC>
struct FwdSimtCfg {
  static constexpr int FT = 2 * FQ;
  static constexpr int QS = SimtCfg<D>::QS, PS = SimtCfg<D>::PS, OC = SimtCfg<D>::OC;
  static constexpr int NKB = ASYNC ? 2 : 1;  // K buffers
  static constexpr int SMEM_BYTES = (FQ * QS + NKB * BK * QS + BK * D + FQ * PS) * 4;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA exceeded");
};

// 16-byte global -> shared copy that bypasses the registers (cp.async); a
// row past T copies nothing and zero-fills (src-size 0)
__device__ __forceinline__ void cp_async16(float* dst, const float* src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// rows [r0, r0 + BK) of a [T][D] fp32 matrix into smem rows of LS floats
template <int D, int LS, int NT>
__device__ __forceinline__ void load_tile_async(float* dst, const float* src, int r0, int T) {
  constexpr int V = D / 4;
#pragma unroll 4
  for (int idx = threadIdx.x; idx < BK * V; idx += NT) {
    const int r = idx / V, c4 = idx % V;
    const bool valid = r0 + r < T;
    cp_async16(dst + r * LS + 4 * c4,
               valid ? src + static_cast<size_t>(r0 + r) * D + 4 * c4 : src, valid);
  }
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename Tin, int D, int FQ, bool ASYNC>
__global__ void __launch_bounds__(2 * FQ)
    fa_fwd_simt_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                       const Tin* __restrict__ v, Tin* __restrict__ o, float* __restrict__ lse,
                       int B, int Hq, int Hkv, int T, float scale, int wl, int wr,
                       const uint32_t* __restrict__ lg_bits, int lg_causal) {
  using C = FwdSimtCfg<D, FQ, ASYNC>;
  constexpr int QS = C::QS, PS = C::PS, OC = C::OC, FT = C::FT;
  constexpr int GW = D >= 64 ? 4 : (D == 32 ? 2 : 1);  // contiguous output columns
  extern __shared__ float4 smem4[];
  float* sQ = reinterpret_cast<float*>(smem4);
  float* sK0 = sQ + FQ * QS;  // K buffer(s)
  float* sV = sK0 + C::NKB * BK * QS;
  float* sP = sV + BK * D;

  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int BH = B * Hq;
  const int n_qt = (T + FQ - 1) / FQ;
  const int n_kt = (T + BK - 1) / BK;
  const int qt = n_qt - 1 - static_cast<int>(blockIdx.x / BH);  // last (causal: longest) first
  const int bh = static_cast<int>(blockIdx.x % BH);
  const int b = bh / Hq, h = bh - (bh / Hq) * Hq;
  const int hk = h / (Hq / Hkv);
  const int q0 = qt * FQ;
  const size_t qoff = static_cast<size_t>(bh) * T * D;
  const size_t kvoff = static_cast<size_t>(b * Hkv + hk) * T * D;

  load_tile<D, QS, FQ, FT>(sQ, q + qoff, q0, T);

  float m[8], lp[8], acc[8][OC];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    m[i] = -INFINITY;
    lp[i] = 0.f;
#pragma unroll
    for (int c = 0; c < OC; ++c) acc[i][c] = 0.f;
  }

  // KV blocks holding keys [q0 - wl, q0 + FQ - 1 + wr] of the band, within T
  const int b_lo = wl < 0 ? 0 : max(0, q0 - wl) / BK;
  const int b_hi = wr < 0 ? n_kt : min(n_kt, min(T - 1, q0 + FQ - 1 + wr) / BK + 1);
  // local-global: global keys may sit in any block (before the rows' last
  // key when causal); blocks with neither band keys nor global keys are skipped
  const int j_lo = lg_bits ? 0 : b_lo;
  const int j_hi = lg_bits ? (lg_causal ? min(n_kt, min(T - 1, q0 + FQ - 1) / BK + 1) : n_kt)
                           : b_hi;
  // ASYNC: K(j_lo) and V(j_lo) in flight before the loop (two commit groups)
  if constexpr (ASYNC) {
    if (j_lo < j_hi) {
      load_tile_async<D, QS, FT>(sK0, reinterpret_cast<const float*>(k) + kvoff, j_lo * BK, T);
      cp_async_commit();
      load_tile_async<D, D, FT>(sV, reinterpret_cast<const float*>(v) + kvoff, j_lo * BK, T);
      cp_async_commit();
    }
  }
  for (int j = j_lo; j < j_hi; ++j) {
    float* sK = sK0;
    if constexpr (ASYNC) {
      // in flight: K(j), V(j); K(j) is the older group
      sK = sK0 + ((j - j_lo) & 1) * (BK * QS);  // K(j_lo) went to buffer 0
      cp_async_wait<1>();
      __syncthreads();
      // the other K buffer was last read by S(j - 1), finished before the
      // barrier that preceded P.V(j - 1)
      if (j + 1 < j_hi)
        load_tile_async<D, QS, FT>(sK0 + ((j + 1 - j_lo) & 1) * (BK * QS),
                                   reinterpret_cast<const float*>(k) + kvoff, (j + 1) * BK, T);
      cp_async_commit();  // (an empty group on the last block keeps the count)
    } else {
      if (lg_bits && (j < b_lo || j >= b_hi) &&
          (__ldg(lg_bits + 2 * j) | __ldg(lg_bits + 2 * j + 1)) == 0u)
        continue;
      __syncthreads();  // previous block's K, V, P no longer in use
      load_tile<D, QS, BK, FT>(sK, k + kvoff, j * BK, T);
      load_tile<D, D, BK, FT>(sV, v + kvoff, j * BK, T);
      __syncthreads();
    }

    // S = Q K^T for the thread's 8 x 4 scores
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) s[i][c] = 0.f;
#pragma unroll 2
    for (int kk = 0; kk < D; kk += 4) {
      float4 kv[4];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        kv[c] = *reinterpret_cast<const float4*>(sK + (tx * 4 + c) * QS + kk);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 qv = *reinterpret_cast<const float4*>(sQ + (ty * 8 + i) * QS + kk);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          s[i][c] = fmaf(qv.x, kv[c].x, s[i][c]);
          s[i][c] = fmaf(qv.y, kv[c].y, s[i][c]);
          s[i][c] = fmaf(qv.z, kv[c].z, s[i][c]);
          s[i][c] = fmaf(qv.w, kv[c].w, s[i][c]);
        }
      }
    }

    // scale, mask, online softmax update in log2 units: the running maximum
    // m is a rounded scaled score (times log2(e)), and every exponent
    // argument s * scale log2(e) - m is formed by one fused multiply-add, so
    // m's own rounding cancels between l and L = (m + log2 l) ln 2.
    const float sl2 = scale * 1.4426950408889634f;
    const int kb = j * BK + tx * 4;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = q0 + ty * 8 + i;
      bool keep[4];
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int key = kb + c;
        keep[c] = key < T && (wr < 0 || key <= row + wr) && (wl < 0 || key >= row - wl);
        if (lg_bits && !keep[c] && key < T && (!lg_causal || key <= row))
          keep[c] = ((__ldg(lg_bits + (key >> 5)) >> (key & 31)) & 1u) != 0u;
        if (keep[c]) mx = fmaxf(mx, s[i][c] * sl2);
      }
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m[i], mx);
      const float mo = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = ex2_approx(m[i] - mo);  // 0 while m[i] = -inf
      float p[4], ps = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        p[c] = keep[c] ? ex2_approx(fmaf(s[i][c], sl2, -mo)) : 0.f;
        ps += p[c];
      }
      lp[i] = lp[i] * alpha + ps;
#pragma unroll
      for (int c = 0; c < OC; ++c) acc[i][c] *= alpha;
      m[i] = m_new;
      *reinterpret_cast<float4*>(sP + (ty * 8 + i) * PS + tx * 4) = make_float4(p[0], p[1], p[2], p[3]);
    }
    if constexpr (ASYNC) cp_async_wait<1>();  // V(j): only K(j + 1) may still be in flight
    __syncthreads();

    // O += P V
#pragma unroll 2
    for (int kk = 0; kk < BK; kk += 4) {
      float4 pv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) pv[i] = *reinterpret_cast<const float4*>(sP + (ty * 8 + i) * PS + kk);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float vv[OC];
        const float* vr = sV + (kk + u) * D;
#pragma unroll
        for (int c = 0; c < OC; c += GW) {
          if constexpr (GW == 4) {
            const float4 t4 = *reinterpret_cast<const float4*>(vr + ocol<D>(tx, c));
            vv[c] = t4.x; vv[c + 1] = t4.y; vv[c + 2] = t4.z; vv[c + 3] = t4.w;
          } else if constexpr (GW == 2) {
            const float2 t2 = *reinterpret_cast<const float2*>(vr + ocol<D>(tx, c));
            vv[c] = t2.x; vv[c + 1] = t2.y;
          } else {
            vv[c] = vr[ocol<D>(tx, c)];
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float pu = u == 0 ? pv[i].x : (u == 1 ? pv[i].y : (u == 2 ? pv[i].z : pv[i].w));
#pragma unroll
          for (int c = 0; c < OC; ++c) acc[i][c] = fmaf(pu, vv[c], acc[i][c]);
        }
      }
    }
    if constexpr (ASYNC) {
      // V(j + 1) into the V buffer once every thread is done with V(j) and P
      __syncthreads();
      if (j + 1 < j_hi)
        load_tile_async<D, D, FT>(sV, reinterpret_cast<const float*>(v) + kvoff, (j + 1) * BK, T);
      cp_async_commit();
    }
  }
  if constexpr (ASYNC) cp_async_wait<0>();

  // normalise and store
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float l = lp[i];
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    const int row = q0 + ty * 8 + i;
    if (row < T) {
      const float inv = 1.f / l;
      Tin* orow = o + qoff + static_cast<size_t>(row) * D;
#pragma unroll
      for (int c = 0; c < OC; c += GW) {
        float y[4];
#pragma unroll
        for (int e = 0; e < GW; ++e) y[e] = acc[i][c + e] * inv;
        store_out(orow + ocol<D>(tx, c), y, GW);
      }
      if (tx == 0) lse[static_cast<size_t>(bh) * T + row] = (m[i] + log2f(l)) * 0.6931471805599453f;
    }
  }
}

template <typename Tin, int D, int FQ, bool ASYNC>
fa_status launch_simt_impl2(const FwdArgs& a) {
  using C = FwdSimtCfg<D, FQ, ASYNC>;
  auto kern = fa_fwd_simt_kernel<Tin, D, FQ, ASYNC>;
  static bool attr_done[64] = {};  // per instantiation and device; benign race
  bool* done = device_flag(attr_done);
  if (done == nullptr || !*done) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return cuda_status(e);
    if (done != nullptr) *done = true;
  }
  const long long blocks = static_cast<long long>(a.B) * a.Hq * ((a.T + FQ - 1) / FQ);
  int wl, wr;
  effective_window(a, wl, wr);
  kern<<<static_cast<unsigned>(blocks), C::FT, C::SMEM_BYTES, a.stream>>>(
      static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v),
      static_cast<Tin*>(a.o), a.lse, a.B, a.Hq, a.Hkv, a.T, a.scale, wl, wr,
      a.local_global ? a.lg_bits : nullptr, a.causal);
  return cuda_status(cudaGetLastError());
}

// the pipelined form for fp32 inputs without a local-global mask, except at
// d = 64 with 128-row CTAs: there its second K buffer (121 KB of shared
// memory instead of 103) leaves room for one CTA per SM instead of two, which
// measured slower (27 vs 31 TFLOP/s at B64 T4096)
template <typename Tin, int D, int FQ>
fa_status launch_simt_impl(const FwdArgs& a) {
  if constexpr (std::is_same<Tin, float>::value && !(D == 64 && FQ == 128))
    if (!a.local_global) return launch_simt_impl2<Tin, D, FQ, true>(a);
  return launch_simt_impl2<Tin, D, FQ, false>(a);
}

// 128-row CTAs (eight warps) for d >= 64 when they still give every SM a CTA;
// 64-row CTAs otherwise (measured: at d <= 32 and for few (b, h) the smaller
// CTA is faster)
template <typename Tin>
fa_status launch_simt_t(const FwdArgs& a) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const bool wide = a.d >= 64 && static_cast<long long>(a.B) * a.Hq * ((a.T + 127) / 128) >= sms;
  switch (a.d) {
    case 16: return launch_simt_impl<Tin, 16, 64>(a);
    case 32: return launch_simt_impl<Tin, 32, 64>(a);
    case 64: return wide ? launch_simt_impl<Tin, 64, 128>(a) : launch_simt_impl<Tin, 64, 64>(a);
    case 128: return wide ? launch_simt_impl<Tin, 128, 128>(a) : launch_simt_impl<Tin, 128, 64>(a);
    default: return FA_ERR_UNSUPPORTED;
  }
}

}  // namespace

fa_status launch_simt(const FwdArgs& a) {
  if (a.dtype == FA_DTYPE_F32) return launch_simt_t<float>(a);
  if (a.dtype == FA_DTYPE_BF16) return launch_simt_t<__nv_bfloat16>(a);
  if (a.dtype == FA_DTYPE_F16) return launch_simt_t<__half>(a);
  return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
