// fa_bwd_tc.cu -- attention backward on tcgen05 tensor cores (bf16 / fp16, sm_103a).
//
// What it computes: the gradients of O = softmax(scale Q K^T + mask) V with
// respect to Q, K and V for an upstream gradient dO, recomputing P from the
// forward's log-sum-exp instead of storing it ("Flash Attention Memory
// Optimization Explained", section "Key Mechanisms", item "Backward
// Checkpointing"):
//   P = exp2(scale log2(e) S - lse log2(e)),  dP = dO V^T,
//   dS = P (dP - D)  with  D_i = sum_c dO[i][c] O[i][c],
//   dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K
// (the softmax Jacobian times the scale of S; the scale is applied once to
// the dK and dQ accumulators in the epilogues).  -D and -lse log2(e) come
// from the preparation kernel (fa_bwd_simt.cu) in a workspace whose rows are
// padded to a multiple of 128 per head (padded rows: -D = 0,
// -lse log2(e) = -inf, so P = 0).  The per-element arithmetic runs on pairs
// of fp32 values (paired FMA, add and multiply).
//
// Two kernels, so that no gradient is accumulated across CTAs by atomics and
// results are deterministic (S and dP are recomputed by both):
//
// fa_bwd_dkdv_tc_kernel -- unit = 128 keys of one (b, KV head).  K and V stay
//   in shared memory; the unit walks the query heads of its group and their
//   64-row query steps inside the band.  Per step i (buffers i & 1):
//     S^T = K Q_i^T, dP^T = V dO_i^T           (SS MMAs, M = 128 keys, N = 64)
//     compute warps: P^T, dS^T (one thread per key = TMEM lane), written back
//       as bf16 over the first 32 columns of the S^T and dP^T buffers
//     dV += P^T dO_i, dK += dS^T Q_i           (TS MMAs, A from TMEM, N = d)
//   While the compute warps work on step i the tensor core already runs the
//   S^T and dP^T of step i + 1.  TMEM: S^T [0,64) [64,128), dP^T [128,192)
//   [192,256), dV [256,256+d), dK [384,384+d).
//
// fa_bwd_dq_tc_kernel -- unit = 128 query rows of one (b, h); walks the KV
//   tiles of the band.  Per KV tile j (S buffer j & 1):
//     S = Q K_j^T, dP = dO V_j^T                (SS MMAs, M = N = 128)
//     compute warps: read dP whole (then the next dP may overwrite it), then
//       S in 32-column chunks; dS (bf16) over the first 64 S columns
//     dQ += dS K_j                              (TS MMA, K_j as MN-major B)
//   TMEM: S [0,128) [128,256), dP [256,384), dQ [384,384+d).
//
// Both grids are persistent (one CTA per SM), units dealt in zig-zag rounds
// longest first; warps 0-3 compute, warp 4 loads (TMA), warp 5 issues MMAs
// (all 32 lanes run its loop so that operands stay warp-uniform; one elected
// lane issues).
// Every wait is bounded (wait.cuh); on expiry the kernel records an error bit,
// drains its own copies and MMAs, frees tensor memory and exits.
#include <cmath>

#include "fa_internal.h"
#include "ptx.cuh"
#include "row_store.cuh"
#include "tc_layout.cuh"
#include "wait.cuh"

namespace fa {

static __device__ unsigned int g_bwd_err;

namespace {

enum : int { kBwdMaskNone = 0, kBwdMaskCausal = 1, kBwdMaskBand = 2, kBwdMaskLocalGlobal = 3 };

constexpr int kBwdThreads = 192;  // compute warps 0-3, producer 4, MMA 5

__device__ __forceinline__ int bwd_unit_index(int k) {
  const int G = static_cast<int>(gridDim.x), bid = static_cast<int>(blockIdx.x);
  return k * G + ((k & 1) ? G - 1 - bid : bid);
}

// the band of the mask kind (a negative side: unbounded)
template <int MASK>
__device__ __forceinline__ void mask_window(int window_left, int window_right, int& wl, int& wr) {
  constexpr bool kBand = MASK == kBwdMaskBand || MASK == kBwdMaskLocalGlobal;
  wl = kBand ? window_left : -1;
  wr = kBand ? window_right : (MASK == kBwdMaskCausal ? 0 : -1);
}

// Paired fp32 multiply (one 64-bit register pair), as ptx::fma2 / ptx::add2.
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// a bounded barrier wait by every lane of a warp, with a warp-uniform result
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned int* err, unsigned int code) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, err, code));
}

// ============================================================ dK, dV kernel
template <int D>
struct KvCfg {
  using TK = TcTile<D, 128>;  // K, V tiles
  using TQ = TcTile<D, 64>;   // Q, dO steps
  static constexpr int NQS = 4;                                   // query-step stages
  static constexpr int STAGE = 2 * TQ::TILE_BYTES + 1024;         // Q, dO, lse2[64], D[64]
  static constexpr int SMEM_BYTES = 1024 + 2 * TK::TILE_BYTES + NQS * STAGE + 256;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA exceeded");
  static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 384;
};

// query steps (64 rows) of KV tile j: queries [kb - wr, kb + 127 + wl] in [0, T)
__device__ __forceinline__ void kv_query_range(int kb, int T, int wl, int wr, int& lo, int& hi) {
  const int nq = (T + 63) >> 6;
  lo = wr < 0 ? 0 : max(0, kb - wr) >> 6;
  const long long last = wl < 0 ? static_cast<long long>(T) - 1
                                : min(static_cast<long long>(T) - 1,
                                      static_cast<long long>(kb) + 127 + wl);
  hi = min(nq, static_cast<int>(last >> 6) + 1);
  if (hi < lo) hi = lo;
}

// Local-global masks: a KV tile that holds a global key is attended by every
// query (from the key on when causal), so its query steps run to the end.
__device__ __forceinline__ void kv_query_range_lg(int kb, int T, int wl, int wr,
                                                  const uint32_t* lg_bits, int causal, int& lo,
                                                  int& hi) {
  kv_query_range(kb, T, wl, wr, lo, hi);
  const uint4 g = __ldg(reinterpret_cast<const uint4*>(lg_bits) + (kb >> 7));
  const uint32_t w[4] = {g.x, g.y, g.z, g.w};
  int first = -1;  // first global key of the tile
#pragma unroll
  for (int i = 3; i >= 0; --i)
    if (w[i] != 0u) first = kb + 32 * i + __ffs(static_cast<int>(w[i])) - 1;
  if (first >= 0) {
    lo = causal ? min(lo, first >> 6) : 0;
    hi = (T + 63) >> 6;
  }
}

// Bits e of a 32-column group starting at column `base` with lo <= base + e <= hi.
__device__ __forceinline__ uint32_t range_bits32(int lo, int hi, int base) {
  const int a = max(lo - base, 0), b = min(hi - base, 31);
  if (a > b) return 0u;
  const uint32_t upto_b = b >= 31 ? 0xffffffffu : ((1u << (b + 1)) - 1u);
  return upto_b & ~((1u << a) - 1u);
}

template <int D, int MASK, bool F16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmdO,
                          const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV,
                          const float* __restrict__ delta, const float* __restrict__ lse2,
                          uint16_t* __restrict__ dK, uint16_t* __restrict__ dV, int B, int Hq,
                          int Hkv, int T, int Tp, float scale, float scale_log2, int num_units,
                          int window_left, int window_right, const uint32_t* __restrict__ lg_bits,
                          int lg_causal) {
  constexpr bool LG = MASK == kBwdMaskLocalGlobal;
  using C = KvCfg<D>;
  using TK = typename C::TK;
  using TQ = typename C::TQ;
  constexpr int NQS = C::NQS;
  constexpr uint32_t IDESC_ST = ptx::idesc_16bit(128, 64, false, false, F16);
  constexpr uint32_t IDESC_G = ptx::idesc_16bit(128, D, false, true, F16);
  int wl, wr;
  mask_window<MASK>(window_left, window_right, wl, wr);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sK = sm;
  uint8_t* sV = sK + TK::TILE_BYTES;
  uint8_t* sStage = sV + TK::TILE_BYTES;  // NQS x {Q, dO, lse2, D}
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStage + NQS * C::STAGE);
  uint64_t* bar_kvfull = bars;
  uint64_t* bar_kvempty = bars + 1;
  uint64_t* bar_qfull = bars + 2;          // [NQS]
  uint64_t* bar_qempty = bar_qfull + NQS;  // [NQS]
  uint64_t* bar_sfull = bar_qempty + NQS;  // [2] S^T and dP^T of a step done
  uint64_t* bar_pfull = bar_sfull + 2;     // [2] P^T, dS^T written (4 warp arrivals)
  uint64_t* bar_dkv = bar_pfull + 2;       // the unit's last dK, dV MMA done
  uint64_t* bar_final = bar_dkv + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_final + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_kvfull, 1);
    ptx::mbar_init(bar_kvempty, 1);
    for (int s = 0; s < NQS; ++s) {
      ptx::mbar_init(&bar_qfull[s], 1);
      ptx::mbar_init(&bar_qempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&bar_sfull[b], 1);
      ptx::mbar_init(&bar_pfull[b], 4);
    }
    ptx::mbar_init(bar_dkv, 1);
    ptx::mbar_init(bar_final, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int BHk = B * Hkv;
  const int group = Hq / Hkv;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmdO);
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      const uint64_t pol_first = ptx::policy_evict_first();
      const uint64_t pol_last = ptx::policy_evict_last();
      int nu = 0, ns = 0;  // units and query steps loaded so far
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int idx = bwd_unit_index(k);
        if (idx >= num_units) break;
        const int j = idx / BHk, bhk = idx - (idx / BHk) * BHk;
        const int b = bhk / Hkv, hk = bhk - b * Hkv;
        const int kb = j * 128;
        if (nu > 0 && !wait_bar(bar_kvempty, (nu - 1) & 1, abort_flag, &g_bwd_err, kErrWaitLoad))
          break;
        ptx::mbar_arrive_expect_tx(bar_kvfull, 2 * TK::TILE_BYTES);
#pragma unroll
        for (int bx = 0; bx < TK::NBOX; ++bx) {
          ptx::tma_load_3d_hint(sK + bx * TK::BOX_BYTES, &tmK, bar_kvfull, bx * 64, kb, bhk,
                                pol_first);
          ptx::tma_load_3d_hint(sV + bx * TK::BOX_BYTES, &tmV, bar_kvfull, bx * 64, kb, bhk,
                                pol_first);
        }
        ++nu;
        int qlo, qhi;
        if constexpr (LG) kv_query_range_lg(kb, T, wl, wr, lg_bits, lg_causal, qlo, qhi);
        else kv_query_range(kb, T, wl, wr, qlo, qhi);
        for (int g = 0; ok && g < group; ++g) {
          const int bh = b * Hq + hk * group + g;
          for (int qt = qlo; qt < qhi; ++qt) {
            const int st = ns % NQS;
            if (ns >= NQS && !wait_bar(&bar_qempty[st], ((ns / NQS) - 1) & 1, abort_flag,
                                       &g_bwd_err, kErrWaitLoad)) {
              ok = false;
              break;
            }
            uint8_t* stage = sStage + st * C::STAGE;
            ptx::mbar_arrive_expect_tx(&bar_qfull[st], 2 * TQ::TILE_BYTES + 512);
#pragma unroll
            for (int bx = 0; bx < TQ::NBOX; ++bx) {
              ptx::tma_load_3d_hint(stage + bx * TQ::BOX_BYTES, &tmQ, &bar_qfull[st], bx * 64,
                                    qt * 64, bh, pol_last);
              ptx::tma_load_3d_hint(stage + TQ::TILE_BYTES + bx * TQ::BOX_BYTES, &tmdO,
                                    &bar_qfull[st], bx * 64, qt * 64, bh, pol_last);
            }
            const size_t row = static_cast<size_t>(bh) * Tp + qt * 64;
            ptx::bulk_g2s(stage + 2 * TQ::TILE_BYTES, lse2 + row, 256, &bar_qfull[st]);
            ptx::bulk_g2s(stage + 2 * TQ::TILE_BYTES + 256, delta + row, 256, &bar_qfull[st]);
            ++ns;
          }
        }
      }
      // own copies still in flight (only after an abort) land before exit
      if (nu > 0) drain_bar(bar_kvfull, (nu - 1) & 1, &g_bwd_err);
      for (int c = max(0, ns - NQS); c < ns; ++c)
        drain_bar(&bar_qfull[c % NQS], (c / NQS) & 1, &g_bwd_err);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs the issue loop (its branches are warp-uniform:
    // every wait ends in a vote); one elected lane issues the MMAs and
    // commits, so that descriptors and addresses stay warp-uniform values
    {
      const uint32_t aK = ptx::smem_u32(sK), aV = ptx::smem_u32(sV);
      const uint32_t aStage = ptx::smem_u32(sStage);
      int nu = 0, gs = 0;  // units, query steps issued so far
      bool ok = true;
      // dV += P^T dO_s and dK += dS^T Q_s for step s (first: the unit's first step)
      auto grad = [&](int s, int first) -> bool {
        const int bb = s & 1, st = s % NQS;
        if (!wait_all(&bar_pfull[bb], (s >> 1) & 1, abort_flag, &g_bwd_err, kErrWaitMma))
          return false;
        ptx::tc_fence_after();
        const uint32_t q_lo = TQ::mnmajor_lo(aStage + st * C::STAGE);
        const uint32_t do_lo = TQ::mnmajor_lo(aStage + st * C::STAGE + TQ::TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < TQ::PV_KSTEPS; ++kk) {
          const uint32_t acc = (s > first || kk > 0) ? 1u : 0u;
          ptx::mma_ts_lh_e(tmem + C::COL_DV, tmem + C::COL_S + bb * 64 + kk * 8,
                         do_lo + TQ::mnmajor_step(kk), TQ::DESC_HI, IDESC_G, acc);
          ptx::mma_ts_lh_e(tmem + C::COL_DK, tmem + C::COL_DP + bb * 64 + kk * 8,
                         q_lo + TQ::mnmajor_step(kk), TQ::DESC_HI, IDESC_G, acc);
        }
        ptx::mma_commit_e(&bar_qempty[st]);
        return true;
      };
      for (int k = 0; ok; ++k) {
        const int idx = bwd_unit_index(k);
        if (idx >= num_units) break;
        const int j = idx / BHk;
        int qlo, qhi;
        if constexpr (LG) kv_query_range_lg(j * 128, T, wl, wr, lg_bits, lg_causal, qlo, qhi);
        else kv_query_range(j * 128, T, wl, wr, qlo, qhi);
        const int nsteps = group * (qhi - qlo);
        if (!wait_all(bar_kvfull, nu & 1, abort_flag, &g_bwd_err, kErrWaitMma)) break;
        ++nu;
        ptx::tc_fence_after();
        const int first = gs;
        const uint32_t k_lo = TK::kmajor_lo(aK), v_lo = TK::kmajor_lo(aV);
        for (int i = 0; i < nsteps; ++i) {
          const int st = gs % NQS, bb = gs & 1;
          if (!wait_all(&bar_qfull[st], (gs / NQS) & 1, abort_flag, &g_bwd_err, kErrWaitMma)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t q_lo = TQ::kmajor_lo(aStage + st * C::STAGE);
          const uint32_t do_lo = TQ::kmajor_lo(aStage + st * C::STAGE + TQ::TILE_BYTES);
#pragma unroll
          for (int kk = 0; kk < TK::QK_KSTEPS; ++kk) {
            ptx::mma_ss_lh_e(tmem + C::COL_S + bb * 64, k_lo + TK::kmajor_step(kk), TK::DESC_HI,
                           q_lo + TQ::kmajor_step(kk), TQ::DESC_HI, IDESC_ST, kk > 0 ? 1u : 0u);
            ptx::mma_ss_lh_e(tmem + C::COL_DP + bb * 64, v_lo + TK::kmajor_step(kk), TK::DESC_HI,
                           do_lo + TQ::kmajor_step(kk), TQ::DESC_HI, IDESC_ST, kk > 0 ? 1u : 0u);
          }
          ptx::mma_commit_e(&bar_sfull[bb]);
          if (gs > first && !grad(gs - 1, first)) {
            ok = false;
            break;
          }
          ++gs;
        }
        if (ok && nsteps > 0) ok = grad(gs - 1, first);
        ptx::mma_commit_e(bar_kvempty);
        ptx::mma_commit_e(bar_dkv);
      }
      ptx::mma_commit_e(bar_final);
      drain_bar(bar_final, 0, &g_bwd_err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute warps
    const int r = warp * 32 + lane;  // key row of the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    int nu = 0, gs = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int idx = bwd_unit_index(k);
      if (idx >= num_units) break;
      const int j = idx / BHk, bhk = idx - (idx / BHk) * BHk;
      const int kb = j * 128;
      const int key = kb + r;
      int qlo, qhi;
      if constexpr (LG) kv_query_range_lg(kb, T, wl, wr, lg_bits, lg_causal, qlo, qhi);
      else kv_query_range(kb, T, wl, wr, qlo, qhi);
      // local-global: this key is a global key (kept for every query, from
      // the key on when causal)
      bool kglob = false;
      if constexpr (LG) kglob = key < T && ((__ldg(lg_bits + (key >> 5)) >> (key & 31)) & 1u);
      const int nsteps = group * (qhi - qlo);
      for (int i = 0; i < nsteps; ++i, ++gs) {
        const int st = gs % NQS, bb = gs & 1;
        const int q0 = (qlo + i % (qhi - qlo)) * 64;
        // S^T and dP^T of the step; the stage's lse2 and D rows (bulk copies
        // that complete on the stage's barrier, which these warps observe too)
        ok = __all_sync(0xffffffffu, wait_bar(&bar_sfull[bb], (gs >> 1) & 1, abort_flag,
                                              &g_bwd_err, kErrWaitSoftmax) &&
                                         wait_bar(&bar_qfull[st], (gs / NQS) & 1, abort_flag,
                                                  &g_bwd_err, kErrWaitSoftmax));
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t s0[32], s1[32], p0[32], p1[32];
        ptx::tmem_ld32(tmem + lane_off + C::COL_S + bb * 64, s0);
        ptx::tmem_ld32(tmem + lane_off + C::COL_S + bb * 64 + 32, s1);
        ptx::tmem_ld32(tmem + lane_off + C::COL_DP + bb * 64, p0);
        ptx::tmem_ld32(tmem + lane_off + C::COL_DP + bb * 64 + 32, p1);
        ptx::tmem_ld_wait(s0);
        ptx::reg_fence(s1);
        ptx::reg_fence(p0);
        ptx::reg_fence(p1);
        const float* l2s = reinterpret_cast<const float*>(sStage + st * C::STAGE +
                                                          2 * TQ::TILE_BYTES);
        const float* dls = l2s + 64;  // (l2s: -lse log2(e) per query; dls: -D)
        // the tile needs the mask unless every (key, query) pair lies in the band
        const bool inside = (wr < 0 || kb + 127 <= q0 + wr) && (wl < 0 || kb >= q0 + 63 - wl);
        int c_lo = wr < 0 ? 0 : key - wr - q0;  // first kept query column
        int c_hi = wl < 0 ? 63 : key + wl - q0;  // last kept query column
        if (LG && kglob) {
          // a global key: the band widens to every query (from the key on)
          c_lo = lg_causal ? key - q0 : 0;
          c_hi = 63;
        }
        // P^T = 2^(s scale log2(e) - lse log2(e)) and dS^T = P^T (dP^T - D) for two
        // query columns at a time; the columns' -lse log2(e) and -D come from the
        // stage as 8-byte shared loads
        const uint64_t sl2x2 = ptx::f2_pack(scale_log2, scale_log2);
        uint32_t pp[32], dd[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t(&sv)[32] = h == 0 ? s0 : s1;
          const uint32_t(&dv)[32] = h == 0 ? p0 : p1;
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int c = h * 32 + e;
            const uint64_t nl2 = *reinterpret_cast<const uint64_t*>(l2s + c);
            const uint64_t nd = *reinterpret_cast<const uint64_t*>(dls + c);
            const uint64_t x2 = ptx::fma2(
                ptx::f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sl2x2, nl2);
            float x0, x1;
            ptx::f2_unpack(x2, x0, x1);
            if (!inside) {
              if (c < c_lo || c > c_hi) x0 = -INFINITY;
              if (c + 1 < c_lo || c + 1 > c_hi) x1 = -INFINITY;
            }
            const float pa = ptx::ex2(x0), pb = ptx::ex2(x1);
            const uint64_t t2 = ptx::add2(
                ptx::f2_pack(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])), nd);
            float da, db;
            ptx::f2_unpack(mul2(ptx::f2_pack(pa, pb), t2), da, db);
            pp[h * 16 + e / 2] = ptx::pack_x2<F16>(pa, pb);
            dd[h * 16 + e / 2] = ptx::pack_x2<F16>(da, db);
          }
        }
        ptx::tmem_st32(tmem + lane_off + C::COL_S + bb * 64, pp);
        ptx::tmem_st32(tmem + lane_off + C::COL_DP + bb * 64, dd);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bar_pfull[bb]);
      }
      if (!ok) break;
      // ---- epilogue: dV and dK rows of this key (dK times the scale of S)
      ok = __all_sync(0xffffffffu,
                      wait_bar(bar_dkv, nu & 1, abort_flag, &g_bwd_err, kErrWaitEpilogue));
      ++nu;
      if (!ok) break;
      ptx::tc_fence_after();
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        // rows of the lane pair, written as whole 32-byte sectors (row_store.cuh)
        const RowPair rp = row_pair((which == 0 ? dV : dK) + static_cast<size_t>(bhk) * T * D, D,
                                    key, T, lane);
        const uint32_t col = which == 0 ? C::COL_DV : C::COL_DK;
        const float sc = which == 0 ? 1.f : scale;
        if constexpr (D >= 32) {
#pragma unroll
          for (int oc = 0; oc < D / 32; ++oc) {
            uint32_t o[32];
            ptx::tmem_ld32(tmem + lane_off + col + oc * 32, o);
            ptx::tmem_ld_wait(o);
            uint32_t pk[16];
#pragma unroll
            for (int v = 0; v < 16; ++v)
              pk[v] = ptx::pack_x2<F16>(__uint_as_float(o[2 * v]) * sc,
                                        __uint_as_float(o[2 * v + 1]) * sc);
            store_sector_pair(rp, oc * 32, pk);
            store_sector_pair(rp, oc * 32 + 16, pk + 8);
          }
        } else {
          uint32_t o[16];
          ptx::tmem_ld16(tmem + lane_off + col, o);
          ptx::tmem_ld_wait(o);
          uint32_t pk[8];
#pragma unroll
          for (int v = 0; v < 8; ++v)
            pk[v] = ptx::pack_x2<F16>(__uint_as_float(o[2 * v]) * sc,
                                      __uint_as_float(o[2 * v + 1]) * sc);
          store_sector_pair(rp, 0, pk);
        }
      }
      // the dK, dV reads are complete before this warp releases its next P^T
      ptx::tc_fence_before();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 0) ptx::tmem_dealloc(tmem, 512);
}

// ============================================================ dQ kernel
template <int D>
struct QCfg {
  using TT = TcTile<D, 128>;
  static constexpr int NSK = D == 128 ? 3 : 4;
  static constexpr int NSV = D == 128 ? 2 : 4;
  static constexpr int SMEM_BYTES = 1024 + (2 + NSK + NSV) * TT::TILE_BYTES + 256;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA exceeded");
  static constexpr uint32_t COL_S = 0, COL_DP = 256, COL_DQ = 384;
};

template <int D, int MASK, bool F16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmdO,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const float* __restrict__ delta, const float* __restrict__ lse2,
                        uint16_t* __restrict__ dQ, int B, int Hq, int Hkv, int T, int Tp,
                        float scale, float scale_log2, int num_units, int window_left,
                        int window_right, const uint32_t* __restrict__ lg_bits,
                        const int* __restrict__ lg_list, const int* __restrict__ lg_count,
                        int lg_causal) {
  constexpr bool LG = MASK == kBwdMaskLocalGlobal;
  using C = QCfg<D>;
  using TT = typename C::TT;
  constexpr int NSK = C::NSK, NSV = C::NSV;
  constexpr int TILE = TT::TILE_BYTES;
  constexpr uint32_t IDESC_S = ptx::idesc_16bit(128, 128, false, false, F16);
  constexpr uint32_t IDESC_DQ = ptx::idesc_16bit(128, D, false, true, F16);
  int wl, wr;
  mask_window<MASK>(window_left, window_right, wl, wr);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = sm;
  uint8_t* sdO = sQ + TILE;
  uint8_t* sK = sdO + TILE;  // NSK
  uint8_t* sV = sK + NSK * TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + NSV * TILE);
  uint64_t* bar_qfull = bars;
  uint64_t* bar_qempty = bars + 1;
  uint64_t* bar_kfull = bars + 2;        // [NSK]
  uint64_t* bar_kempty = bar_kfull + NSK;
  uint64_t* bar_vfull = bar_kempty + NSK;  // [NSV]
  uint64_t* bar_vempty = bar_vfull + NSV;
  uint64_t* bar_sfull = bar_vempty + NSV;  // [2] S and dP of a KV tile done
  uint64_t* bar_dpfree = bar_sfull + 2;    // dP read by the compute warps (4 arrivals)
  uint64_t* bar_pfull = bar_dpfree + 1;    // [2] dS written (4 arrivals)
  uint64_t* bar_dq = bar_pfull + 2;        // the unit's last dQ MMA done
  uint64_t* bar_final = bar_dq + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_final + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_qfull, 1);
    ptx::mbar_init(bar_qempty, 1);
    for (int s = 0; s < NSK; ++s) {
      ptx::mbar_init(&bar_kfull[s], 1);
      ptx::mbar_init(&bar_kempty[s], 1);
    }
    for (int s = 0; s < NSV; ++s) {
      ptx::mbar_init(&bar_vfull[s], 1);
      ptx::mbar_init(&bar_vempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&bar_sfull[b], 1);
      ptx::mbar_init(&bar_pfull[b], 4);
    }
    ptx::mbar_init(bar_dpfree, 4);
    ptx::mbar_init(bar_dq, 1);
    ptx::mbar_init(bar_final, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int BH = B * Hq;
  const int n_qb = (T + 127) >> 7;
  // unit idx: row block (last first: the longest when causal) and (b, h); its
  // KV tiles are the band's [lo, hi) and, for local-global masks, the nb tiles
  // holding a global key below lo plus those from list index ia up to the
  // unit's last row (cnt tiles in all)
  auto unit_of = [&](int idx, int& q0, int& bh, int& lo, int& hi, int& cnt, int& nb, int& ia) {
    q0 = (n_qb - 1 - idx / BH) * 128;
    bh = idx - (idx / BH) * BH;
    lo = wl < 0 ? 0 : max(0, q0 - wl) >> 7;
    const long long last = wr < 0 ? static_cast<long long>(T) - 1
                                  : min(static_cast<long long>(T) - 1,
                                        static_cast<long long>(q0) + 127 + wr);
    hi = static_cast<int>(last >> 7) + 1;
    cnt = hi - lo;
    nb = ia = 0;
    if constexpr (LG) {
      const int n = __ldg(lg_count);
      const int cap = lg_causal ? min(T - 1, q0 + 127) >> 7 : (T - 1) >> 7;
      auto lower_bound = [&](int x) {
        int a = 0, b = n;
        while (a < b) {
          const int mid = (a + b) >> 1;
          if (__ldg(lg_list + mid) < x) a = mid + 1;
          else b = mid;
        }
        return a;
      };
      nb = lower_bound(lo);
      ia = lower_bound(hi);
      cnt += nb + max(0, lower_bound(cap + 1) - ia);
    }
  };
  // KV tile of the unit's jj-th visited tile
  auto tile_of = [&](int lo, int hi, int nb, int ia, int jj) -> int {
    if constexpr (!LG) {
      return lo + jj;
    } else {
      if (jj < nb) return __ldg(lg_list + jj);
      if (jj < nb + (hi - lo)) return lo + (jj - nb);
      return __ldg(lg_list + ia + (jj - nb - (hi - lo)));
    }
  };

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmdO);
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      const uint64_t pol_first = ptx::policy_evict_first();
      const uint64_t pol_last = ptx::policy_evict_last();
      int nu = 0, kc = 0, vc = 0;  // units, K tiles, V tiles loaded so far
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int idx = bwd_unit_index(k);
        if (idx >= num_units) break;
        int q0, bh, lo, hi, cnt, nb, ia;
        unit_of(idx, q0, bh, lo, hi, cnt, nb, ia);
        const int b = bh / Hq, h = bh - b * Hq;
        const int zkv = b * Hkv + h / (Hq / Hkv);
        if (nu > 0 && !wait_bar(bar_qempty, (nu - 1) & 1, abort_flag, &g_bwd_err, kErrWaitLoad))
          break;
        ptx::mbar_arrive_expect_tx(bar_qfull, 2 * TILE);
#pragma unroll
        for (int bx = 0; bx < TT::NBOX; ++bx) {
          ptx::tma_load_3d_hint(sQ + bx * TT::BOX_BYTES, &tmQ, bar_qfull, bx * 64, q0, bh,
                                pol_first);
          ptx::tma_load_3d_hint(sdO + bx * TT::BOX_BYTES, &tmdO, bar_qfull, bx * 64, q0, bh,
                                pol_first);
        }
        ++nu;
        for (int jj = 0; jj < cnt; ++jj) {
          const int j = tile_of(lo, hi, nb, ia, jj);
          const int sk = kc % NSK, sv = vc % NSV;
          if (kc >= NSK && !wait_bar(&bar_kempty[sk], ((kc / NSK) - 1) & 1, abort_flag,
                                     &g_bwd_err, kErrWaitLoad)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&bar_kfull[sk], TILE);
#pragma unroll
          for (int bx = 0; bx < TT::NBOX; ++bx)
            ptx::tma_load_3d_hint(sK + sk * TILE + bx * TT::BOX_BYTES, &tmK, &bar_kfull[sk],
                                  bx * 64, j * 128, zkv, pol_last);
          ++kc;
          if (vc >= NSV && !wait_bar(&bar_vempty[sv], ((vc / NSV) - 1) & 1, abort_flag,
                                     &g_bwd_err, kErrWaitLoad)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&bar_vfull[sv], TILE);
#pragma unroll
          for (int bx = 0; bx < TT::NBOX; ++bx)
            ptx::tma_load_3d_hint(sV + sv * TILE + bx * TT::BOX_BYTES, &tmV, &bar_vfull[sv],
                                  bx * 64, j * 128, zkv, pol_last);
          ++vc;
        }
      }
      // own copies still in flight (only after an abort) land before exit
      if (nu > 0) drain_bar(bar_qfull, (nu - 1) & 1, &g_bwd_err);
      for (int c = max(0, kc - NSK); c < kc; ++c)
        drain_bar(&bar_kfull[c % NSK], (c / NSK) & 1, &g_bwd_err);
      for (int c = max(0, vc - NSV); c < vc; ++c)
        drain_bar(&bar_vfull[c % NSV], (c / NSV) & 1, &g_bwd_err);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs the issue loop (its branches are warp-uniform:
    // every wait ends in a vote); one elected lane issues the MMAs and
    // commits, so that descriptors and addresses stay warp-uniform values
    {
      const uint32_t aQ = ptx::smem_u32(sQ), adO = ptx::smem_u32(sdO);
      const uint32_t aK = ptx::smem_u32(sK), aV = ptx::smem_u32(sV);
      int nu = 0, gs = 0;  // units, KV tiles issued so far (one K and one V per tile)
      bool ok = true;
      // dQ += dS_s K_s for KV tile s (first: the unit's first tile)
      auto grad = [&](int s, int first) -> bool {
        const int bb = s & 1;
        if (!wait_all(&bar_pfull[bb], (s >> 1) & 1, abort_flag, &g_bwd_err, kErrWaitMma))
          return false;
        ptx::tc_fence_after();
        const uint32_t k_lo = TT::mnmajor_lo(aK + (s % NSK) * TILE);
#pragma unroll
        for (int kk = 0; kk < TT::PV_KSTEPS; ++kk)
          ptx::mma_ts_lh_e(tmem + C::COL_DQ, tmem + C::COL_S + bb * 128 + kk * 8,
                         k_lo + TT::mnmajor_step(kk), TT::DESC_HI, IDESC_DQ,
                         (s > first || kk > 0) ? 1u : 0u);
        ptx::mma_commit_e(&bar_kempty[s % NSK]);
        return true;
      };
      for (int k = 0; ok; ++k) {
        const int idx = bwd_unit_index(k);
        if (idx >= num_units) break;
        int q0, bh, lo, hi, cnt, nb, ia;
        unit_of(idx, q0, bh, lo, hi, cnt, nb, ia);
        if (!wait_all(bar_qfull, nu & 1, abort_flag, &g_bwd_err, kErrWaitMma)) break;
        ++nu;
        ptx::tc_fence_after();
        const int first = gs;
        const uint32_t q_lo = TT::kmajor_lo(aQ), do_lo = TT::kmajor_lo(adO);
        for (int jj = 0; jj < cnt; ++jj) {
          const int bb = gs & 1, sk = gs % NSK, sv = gs % NSV;
          if (!wait_all(&bar_kfull[sk], (gs / NSK) & 1, abort_flag, &g_bwd_err, kErrWaitMma)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t k_lo = TT::kmajor_lo(aK + sk * TILE);
#pragma unroll
          for (int kk = 0; kk < TT::QK_KSTEPS; ++kk)
            ptx::mma_ss_lh_e(tmem + C::COL_S + bb * 128, q_lo + TT::kmajor_step(kk), TT::DESC_HI,
                           k_lo + TT::kmajor_step(kk), TT::DESC_HI, IDESC_S, kk > 0 ? 1u : 0u);
          // the dP columns are free once the compute warps have read the last dP
          if (gs > 0 &&
              !wait_all(bar_dpfree, (gs - 1) & 1, abort_flag, &g_bwd_err, kErrWaitMma)) {
            ok = false;
            break;
          }
          if (!wait_all(&bar_vfull[sv], (gs / NSV) & 1, abort_flag, &g_bwd_err, kErrWaitMma)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t v_lo = TT::kmajor_lo(aV + sv * TILE);
#pragma unroll
          for (int kk = 0; kk < TT::QK_KSTEPS; ++kk)
            ptx::mma_ss_lh_e(tmem + C::COL_DP, do_lo + TT::kmajor_step(kk), TT::DESC_HI,
                           v_lo + TT::kmajor_step(kk), TT::DESC_HI, IDESC_S, kk > 0 ? 1u : 0u);
          ptx::mma_commit_e(&bar_vempty[sv]);
          ptx::mma_commit_e(&bar_sfull[bb]);
          if (gs > first && !grad(gs - 1, first)) {
            ok = false;
            break;
          }
          ++gs;
        }
        if (ok && cnt > 0) ok = grad(gs - 1, first);
        ptx::mma_commit_e(bar_qempty);
        ptx::mma_commit_e(bar_dq);
      }
      ptx::mma_commit_e(bar_final);
      drain_bar(bar_final, 0, &g_bwd_err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute warps
    const int r = warp * 32 + lane;  // query row of the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    int nu = 0, gs = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int idx = bwd_unit_index(k);
      if (idx >= num_units) break;
      int q0, bh, lo, hi, cnt, nb, ia;
      unit_of(idx, q0, bh, lo, hi, cnt, nb, ia);
      const int q = q0 + r;
      const size_t wrow = static_cast<size_t>(bh) * Tp + q;  // q < Tp: rows are padded
      // the row's -lse log2(e) and -D, paired for the paired fp32 arithmetic
      const uint64_t nl2x2 = ptx::f2_pack(lse2[wrow], lse2[wrow]);
      const uint64_t ndx2 = ptx::f2_pack(delta[wrow], delta[wrow]);
      const uint64_t sl2x2 = ptx::f2_pack(scale_log2, scale_log2);
      for (int jj = 0; jj < cnt; ++jj, ++gs) {
        const int j = tile_of(lo, hi, nb, ia, jj);
        const int bb = gs & 1;
        ok = __all_sync(0xffffffffu, wait_bar(&bar_sfull[bb], (gs >> 1) & 1, abort_flag,
                                              &g_bwd_err, kErrWaitSoftmax));
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t dp[128];
        ptx::tmem_ld128(tmem + lane_off + C::COL_DP, dp);
        ptx::tmem_ld_wait(dp);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_dpfree);
        const int kb = j * 128;
        // keys at or past T are masked too (their scores are 0, not -inf)
        const bool inside = kb + 127 < T && (wr < 0 || kb + 127 <= q0 + wr) &&
                            (wl < 0 || kb >= q0 + 127 - wl);
        const int hi_c = (wr < 0 ? T - 1 : min(T - 1, q + wr)) - kb;  // last kept column
        const int lo_c = wl < 0 ? -1 : q - wl - kb;                     // first kept column
        // local-global: the tile's global keys (before T, not after the row
        // when causal) are kept as well
        uint4 g4 = make_uint4(0u, 0u, 0u, 0u);
        int ghi_c = -1;
        if constexpr (LG) {
          if (!inside) {
            g4 = __ldg(reinterpret_cast<const uint4*>(lg_bits) + (kb >> 7));
            ghi_c = (lg_causal ? min(T - 1, q) : T - 1) - kb;
          }
        }
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t s[32];
          ptx::tmem_ld32(tmem + lane_off + C::COL_S + bb * 128 + ch * 32, s);
          ptx::tmem_ld_wait(s);
          uint32_t keep = 0xffffffffu;
          if constexpr (LG) {
            const uint32_t gw = ch == 0 ? g4.x : (ch == 1 ? g4.y : (ch == 2 ? g4.z : g4.w));
            if (!inside)
              keep = range_bits32(lo_c, hi_c, 32 * ch) | (gw & range_bits32(0, ghi_c, 32 * ch));
          }
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int c = ch * 32 + e;
            const uint64_t x2 = ptx::fma2(
                ptx::f2_pack(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), sl2x2, nl2x2);
            float x0, x1;
            ptx::f2_unpack(x2, x0, x1);
            if constexpr (LG) {
              if (!((keep >> e) & 1u)) x0 = -INFINITY;
              if (!((keep >> (e + 1)) & 1u)) x1 = -INFINITY;
            } else if (!inside) {
              if (c > hi_c || c < lo_c) x0 = -INFINITY;
              if (c + 1 > hi_c || c + 1 < lo_c) x1 = -INFINITY;
            }
            const float pa = ptx::ex2(x0), pb = ptx::ex2(x1);
            // dS = P (dP - D), two keys at a time
            const uint64_t t2 = ptx::add2(
                ptx::f2_pack(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])), ndx2);
            float da, db;
            ptx::f2_unpack(mul2(ptx::f2_pack(pa, pb), t2), da, db);
            pk[e / 2] = ptx::pack_x2<F16>(da, db);
          }
          // dS chunk ch over columns [16 ch, 16 ch + 16), all already read
          ptx::tmem_st16(tmem + lane_off + C::COL_S + bb * 128 + ch * 16, pk);
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bar_pfull[bb]);
      }
      if (!ok) break;
      // ---- epilogue: the dQ row, times the scale of S
      ok = __all_sync(0xffffffffu,
                      wait_bar(bar_dq, nu & 1, abort_flag, &g_bwd_err, kErrWaitEpilogue));
      ++nu;
      if (!ok) break;
      ptx::tc_fence_after();
      // rows of the lane pair, written as whole 32-byte sectors (row_store.cuh)
      const RowPair rp = row_pair(dQ + static_cast<size_t>(bh) * T * D, D, q, T, lane);
      if constexpr (D >= 32) {
#pragma unroll
        for (int oc = 0; oc < D / 32; ++oc) {
          uint32_t o[32];
          ptx::tmem_ld32(tmem + lane_off + C::COL_DQ + oc * 32, o);
          ptx::tmem_ld_wait(o);
          uint32_t pk[16];
#pragma unroll
          for (int v = 0; v < 16; ++v)
            pk[v] = ptx::pack_x2<F16>(__uint_as_float(o[2 * v]) * scale,
                                      __uint_as_float(o[2 * v + 1]) * scale);
          store_sector_pair(rp, oc * 32, pk);
          store_sector_pair(rp, oc * 32 + 16, pk + 8);
        }
      } else {
        uint32_t o[16];
        ptx::tmem_ld16(tmem + lane_off + C::COL_DQ, o);
        ptx::tmem_ld_wait(o);
        uint32_t pk[8];
#pragma unroll
        for (int v = 0; v < 8; ++v)
          pk[v] = ptx::pack_x2<F16>(__uint_as_float(o[2 * v]) * scale,
                                    __uint_as_float(o[2 * v + 1]) * scale);
        store_sector_pair(rp, 0, pk);
      }
      ptx::tc_fence_before();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 0) ptx::tmem_dealloc(tmem, 512);
}

int bwd_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

template <int D, int MASK, bool F16>
fa_status launch_bwd_tc_impl(const BwdArgs& a) {
  using CK = KvCfg<D>;
  using CQ = QCfg<D>;
  auto kkv = fa_bwd_dkdv_tc_kernel<D, MASK, F16>;
  auto kq = fa_bwd_dq_tc_kernel<D, MASK, F16>;
  static bool attr_done[64] = {};  // per instantiation and device; benign race
  bool* done = device_flag(attr_done);
  if (done == nullptr || !*done) {
    cudaError_t e =
        cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, CK::SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, CQ::SMEM_BYTES);
    if (e != cudaSuccess) return cuda_status(e);
    if (done != nullptr) *done = true;
  }
  using TK = TcTile<D, 128>;
  using TQ = TcTile<D, 64>;
  const long long BH = static_cast<long long>(a.B) * a.Hq;
  const long long BHk = static_cast<long long>(a.B) * a.Hkv;
  CUtensorMap mq64, mdo64, mq, mdo, mk, mv;
  CUresult r;
  if ((r = make_tmap_16bit(&mq64, a.q, D, a.T, BH, TQ::BOX_X, TQ::TMA_SWIZZLE, F16, 64)) !=
          CUDA_SUCCESS ||
      (r = make_tmap_16bit(&mdo64, a.d_o, D, a.T, BH, TQ::BOX_X, TQ::TMA_SWIZZLE, F16, 64)) !=
          CUDA_SUCCESS ||
      (r = make_tmap_16bit(&mq, a.q, D, a.T, BH, TK::BOX_X, TK::TMA_SWIZZLE, F16, 128)) !=
          CUDA_SUCCESS ||
      (r = make_tmap_16bit(&mdo, a.d_o, D, a.T, BH, TK::BOX_X, TK::TMA_SWIZZLE, F16, 128)) !=
          CUDA_SUCCESS ||
      (r = make_tmap_16bit(&mk, a.k, D, a.T, BHk, TK::BOX_X, TK::TMA_SWIZZLE, F16, 128)) !=
          CUDA_SUCCESS ||
      (r = make_tmap_16bit(&mv, a.v, D, a.T, BHk, TK::BOX_X, TK::TMA_SWIZZLE, F16, 128)) !=
          CUDA_SUCCESS)
    return cu_status(r);
  int wl, wr;
  effective_window(a, wl, wr);
  const int Tp = bwd_rows_padded(a.T);
  // scale * log2(e), as in the forward: never exactly 0, so that masked
  // (-inf) exponents never meet a zero factor
  float scale_log2 = a.scale * 1.4426950408889634f;
  if (scale_log2 == 0.f) scale_log2 = 1.17549435e-38f;
  const int sm = bwd_sm_count();
  const long long kv_units = BHk * ((a.T + 127) / 128);
  const long long q_units = BH * ((a.T + 127) / 128);
  kkv<<<static_cast<unsigned>(kv_units < sm ? kv_units : sm), kBwdThreads, CK::SMEM_BYTES,
        a.stream>>>(mq64, mdo64, mk, mv, a.ws_delta, a.ws_lse2, static_cast<uint16_t*>(a.dk),
                    static_cast<uint16_t*>(a.dv), a.B, a.Hq, a.Hkv, a.T, Tp, a.scale, scale_log2,
                    static_cast<int>(kv_units), wl, wr, a.lg_bits, a.causal);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_status(e);
  kq<<<static_cast<unsigned>(q_units < sm ? q_units : sm), kBwdThreads, CQ::SMEM_BYTES,
       a.stream>>>(mq, mdo, mk, mv, a.ws_delta, a.ws_lse2, static_cast<uint16_t*>(a.dq), a.B,
                   a.Hq, a.Hkv, a.T, Tp, a.scale, scale_log2, static_cast<int>(q_units), wl, wr,
                   a.lg_bits, a.lg_list, a.lg_count, a.causal);
  return cuda_status(cudaGetLastError());
}

template <int MASK, bool F16>
fa_status launch_bwd_tc_d(const BwdArgs& a) {
  switch (a.d) {
    case 16: return launch_bwd_tc_impl<16, MASK, F16>(a);
    case 32: return launch_bwd_tc_impl<32, MASK, F16>(a);
    case 64: return launch_bwd_tc_impl<64, MASK, F16>(a);
    case 128: return launch_bwd_tc_impl<128, MASK, F16>(a);
    default: return FA_ERR_UNSUPPORTED;
  }
}

template <bool F16>
fa_status launch_bwd_tc_t(const BwdArgs& a) {
  int wl, wr;
  effective_window(a, wl, wr);
  if (a.local_global) return launch_bwd_tc_d<kBwdMaskLocalGlobal, F16>(a);
  if (wl < 0 && wr < 0) return launch_bwd_tc_d<kBwdMaskNone, F16>(a);
  if (wl < 0 && wr == 0) return launch_bwd_tc_d<kBwdMaskCausal, F16>(a);
  return launch_bwd_tc_d<kBwdMaskBand, F16>(a);
}

}  // namespace

bool bwd_tc_supported(const BwdArgs& a) {
  return a.dtype == FA_DTYPE_BF16 || a.dtype == FA_DTYPE_F16;
}

fa_status launch_bwd_tc(const BwdArgs& a) {
  if (!bwd_tc_supported(a)) return FA_ERR_UNSUPPORTED;
  return a.dtype == FA_DTYPE_F16 ? launch_bwd_tc_t<true>(a) : launch_bwd_tc_t<false>(a);
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
