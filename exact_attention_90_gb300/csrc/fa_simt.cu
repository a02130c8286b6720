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
#include <cmath>

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
template <int D, int FQ>
struct FwdSimtCfg {
  static constexpr int FT = 2 * FQ;
  static constexpr int QS = SimtCfg<D>::QS, PS = SimtCfg<D>::PS, OC = SimtCfg<D>::OC;
  static constexpr int SMEM_BYTES = (FQ * QS + BK * QS + BK * D + FQ * PS) * 4;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA exceeded");
};

template <typename Tin, int D, int FQ>
__global__ void __launch_bounds__(2 * FQ)
    fa_fwd_simt_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                       const Tin* __restrict__ v, Tin* __restrict__ o, float* __restrict__ lse,
                       int B, int Hq, int Hkv, int T, float scale, int wl, int wr,
                       const uint32_t* __restrict__ lg_bits, int lg_causal) {
  using C = FwdSimtCfg<D, FQ>;
  constexpr int QS = C::QS, PS = C::PS, OC = C::OC, FT = C::FT;
  constexpr int GW = D >= 64 ? 4 : (D == 32 ? 2 : 1);  // contiguous output columns
  extern __shared__ float4 smem4[];
  float* sQ = reinterpret_cast<float*>(smem4);
  float* sK = sQ + FQ * QS;
  float* sV = sK + BK * QS;
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
  for (int j = j_lo; j < j_hi; ++j) {
    if (lg_bits && (j < b_lo || j >= b_hi) && (__ldg(lg_bits + 2 * j) | __ldg(lg_bits + 2 * j + 1)) == 0u)
      continue;
    __syncthreads();  // previous block's K, V, P no longer in use
    load_tile<D, QS, BK, FT>(sK, k + kvoff, j * BK, T);
    load_tile<D, D, BK, FT>(sV, v + kvoff, j * BK, T);
    __syncthreads();

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

    // scale, mask, online softmax update.  Natural-log units: the running
    // maximum m is a rounded scaled score, and every exponent argument
    // s * scale - m is formed by one fused multiply-add, so m's own rounding
    // cancels between l and L = m + ln l.
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
        if (keep[c]) mx = fmaxf(mx, s[i][c] * scale);
      }
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m[i], mx);
      const float mo = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = expf(m[i] - mo);  // 0 while m[i] = -inf
      float p[4], ps = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        p[c] = keep[c] ? expf(fmaf(s[i][c], scale, -mo)) : 0.f;
        ps += p[c];
      }
      lp[i] = lp[i] * alpha + ps;
#pragma unroll
      for (int c = 0; c < OC; ++c) acc[i][c] *= alpha;
      m[i] = m_new;
      *reinterpret_cast<float4*>(sP + (ty * 8 + i) * PS + tx * 4) = make_float4(p[0], p[1], p[2], p[3]);
    }
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
  }

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
      if (tx == 0) lse[static_cast<size_t>(bh) * T + row] = m[i] + logf(l);
    }
  }
}

template <typename Tin, int D, int FQ>
fa_status launch_simt_impl(const FwdArgs& a) {
  using C = FwdSimtCfg<D, FQ>;
  auto kern = fa_fwd_simt_kernel<Tin, D, FQ>;
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
