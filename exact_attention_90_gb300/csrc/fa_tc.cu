// fa_tc.cu -- bf16 exact attention forward on tcgen05 tensor cores (sm_103a).
//
// What it computes: for every (batch, query head) and every query row, the
// scaled dot-product attention output O = softmax(scale * Q K^T + mask) V and
// the row log-sum-exp L = m + ln l, without ever writing the T x T score
// matrix to global memory.  Sources (web pages): the yelogs.com Flash
// Attention2/Triton tutorial, section "核心 Kernel 實現" (one program per
// (batch*head, Q block); running m, l and O in fp32; the KV loop stops at the
// diagonal block when causal; O /= l and L = m + log l at the end) and section
// "Softmax 的在線計算" (the recurrence m_new = max(m_old, max s),
// l_new = e^(m_old - m_new) l_old + sum e^(s - m_new)); "Flash Attention
// Memory Optimization Explained", section "Key Mechanisms" (tiles that stay
// on chip, causal look-back only).
//
// How it runs on Blackwell.  One CTA owns 256 query rows of one (b, h) as two
// 128-row tiles Q0, Q1 that share every K/V tile it loads.  Warp roles:
//   warps 0-3 : softmax, correction and epilogue for Q0 (one thread per row)
//   warps 4-7 : the same for Q1
//   warp 8    : TMA producer (Q0, Q1 once; K_j, V_j through an NS-deep ring)
//   warp 9    : MMA issuer (one thread)
//   warps 10-11 complete the third warpgroup, whose registers setmaxnreg
//   hands to the two softmax warpgroups
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   S0 [0,128)  S1 [128,256)  fp32 scores of Q0 K_j^T, Q1 K_j^T
//   P0, P1      bf16 probabilities packed two per column in the first 64
//               columns of S0 / S1 (written by the softmax warps)
//   O0 [256,256+d)  O1 [384,384+d)  fp32 output accumulators
// Per KV tile j the MMA thread issues  PV0_j, S0_{j+1}, PV1_j, S1_{j+1}; while
// the tensor core runs one tile's PV and next S, the other tile's softmax
// warps turn their S into P.  S_{t,j+1} overwrites the columns of P_{t,j};
// it is issued after PV_{t,j} by the same thread, and tcgen05 MMAs of one
// thread execute in issue order.
// The softmax works in the log2 domain (scores times scale*log2(e), exp2 on
// the SFU) and rescales O lazily: the reference maximum is only raised when a
// row's maximum grows by more than 2^8, so most tiles skip the O correction;
// the result is exact because O and l always share the same reference.
#include <cmath>
#include <cstdio>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tc_layout.cuh"
#include "wait.cuh"

namespace fa {

static __device__ unsigned int g_tc_err;

// Tuning parameters (compile-time; defaults are the measured best):
//   FA_TC_P_CHUNKS   -- P is released to the MMA thread in this many pieces
//   FA_TC_REG_SPLIT  -- 1: 384 threads, setmaxnreg moves registers from the
//                       load/MMA warpgroup to the softmax warpgroups;
//                       0: 320 threads, one register budget for all warps
#ifndef FA_TC_P_CHUNKS
#define FA_TC_P_CHUNKS 4
#endif
#ifndef FA_TC_REG_SPLIT
#define FA_TC_REG_SPLIT 1
#endif

template <int D>
struct TcCfg : TcTile<D> {
  using Tile = TcTile<D>;
  static constexpr int NS = D == 128 ? 2 : 4;  // K/V ring depth
  static constexpr int THREADS = FA_TC_REG_SPLIT ? 384 : 320;  // softmax Q0, Q1; load/MMA
  static constexpr int REGS_SOFTMAX = 200;  // per thread after setmaxnreg, warpgroups 0 and 1
  static constexpr int REGS_OTHER = 88;     // warpgroup 2
  static constexpr int P_CHUNKS = FA_TC_P_CHUNKS;  // P released to the MMA in key chunks
  // registers the three warpgroups hold after reallocation
  static constexpr int REGS_SPLIT = FA_TC_REG_SPLIT ? 128 * (2 * REGS_SOFTMAX + REGS_OTHER) : 0;
  static constexpr int SMEM_BYTES = 1024 + (2 + 2 * NS) * Tile::TILE_BYTES + 512;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S0 = 0, COL_O0 = 256;
};

// log2 headroom of the lazy rescale: P values stay below 2^8
#define FA_RESCALE_THRESHOLD 8.0f

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(FA_TC_REG_SPLIT ? 384 : 320, 1)
    fa_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O,
                     float* __restrict__ LSE, int B, int Hq, int Hkv, int T, float scale_log2) {
  using C = TcCfg<D>;
  using Tile = TcTile<D>;
  constexpr int NS = C::NS;
  constexpr int TILE = Tile::TILE_BYTES;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = sm;                  // Q0, Q1
  uint8_t* sK = sm + 2 * TILE;       // NS K tiles
  uint8_t* sV = sK + NS * TILE;      // NS V tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + NS * TILE);
  uint64_t* bar_q = bars;
  uint64_t* bar_kfull = bars + 1;
  uint64_t* bar_vfull = bar_kfull + NS;
  uint64_t* bar_kvempty = bar_vfull + NS;
  uint64_t* bar_sfull = bar_kvempty + NS;  // [2]
  uint64_t* bar_pfull = bar_sfull + 2;     // [2][P_CHUNKS]
  uint64_t* bar_odone = bar_pfull + 2 * C::P_CHUNKS;  // [2]
  uint64_t* bar_final = bar_odone + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_final + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work unit: 256 query rows of one (b, h); longest (last) blocks first
  const int BH = B * Hq;
  const int n_qb = (T + 255) >> 8;
  const int qb = n_qb - 1 - static_cast<int>(blockIdx.x / BH);
  const int bh = static_cast<int>(blockIdx.x % BH);
  const int b = bh / Hq;
  const int h = bh - b * Hq;
  const int hk = h / (Hq / Hkv);
  const int q0 = qb * 256;
  const int n_kv_all = (T + 127) >> 7;
  // KV tiles each Q tile visits (0 if the tile lies past T)
  auto n_of = [&](int t) {
    const int qs = q0 + 128 * t;
    return qs >= T ? 0 : (CAUSAL ? min(n_kv_all, (qs >> 7) + 1) : n_kv_all);
  };
  const int n_t0 = n_of(0), n_t1 = n_of(1);
  const int n_kv = max(n_t0, n_t1);

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_q, 1);
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(&bar_kfull[s], 1);
      ptx::mbar_init(&bar_vfull[s], 1);
      ptx::mbar_init(&bar_kvempty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(&bar_sfull[t], 1);
      for (int c = 0; c < C::P_CHUNKS; ++c) ptx::mbar_init(&bar_pfull[t * C::P_CHUNKS + c], 4);
      ptx::mbar_init(&bar_odone[t], 1);
    }
    ptx::mbar_init(bar_final, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(tmem_slot, C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // every role ends here: all tensor-memory traffic is done before warp 0
  // frees the columns
  auto teardown = [&]() {
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 0) ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  };

  // Each warpgroup's code lives entirely inside its own branch (no code after
  // the branches), so every region compiles under its own register budget.
  if (warp >= 8) {
    // ================================================ warpgroup 2: load, MMA
    if constexpr (FA_TC_REG_SPLIT) ptx::setmaxnreg_dec<C::REGS_OTHER>();
    if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      const uint64_t pol_kv = ptx::policy_evict_last();
      const uint64_t pol_q = ptx::policy_evict_first();
      ptx::mbar_arrive_expect_tx(bar_q, 2 * TILE);
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int bx = 0; bx < Tile::NBOX; ++bx)
          ptx::tma_load_3d_hint(sQ + t * TILE + bx * Tile::BOX_BYTES, &tmQ, bar_q, bx * 64,
                                q0 + 128 * t, bh, pol_q);
      const int zkv = b * Hkv + hk;
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % NS;
        if (j >= NS &&
            !wait_bar(&bar_kvempty[st], ((j / NS) - 1) & 1, abort_flag, &g_tc_err, kErrWaitLoad))
          break;
        ptx::mbar_arrive_expect_tx(&bar_kfull[st], TILE);
#pragma unroll
        for (int bx = 0; bx < Tile::NBOX; ++bx)
          ptx::tma_load_3d_hint(sK + st * TILE + bx * Tile::BOX_BYTES, &tmK, &bar_kfull[st],
                                bx * 64, j * 128, zkv, pol_kv);
        ptx::mbar_arrive_expect_tx(&bar_vfull[st], TILE);
#pragma unroll
        for (int bx = 0; bx < Tile::NBOX; ++bx)
          ptx::tma_load_3d_hint(sV + st * TILE + bx * Tile::BOX_BYTES, &tmV, &bar_vfull[st],
                                bx * 64, j * 128, zkv, pol_kv);
        issued = j + 1;
      }
      // own copies still in flight (only after an abort) land before exit
      drain_bar(bar_q, 0, &g_tc_err);
      for (int j = max(0, issued - NS); j < issued; ++j) {
        drain_bar(&bar_kfull[j % NS], (j / NS) & 1, &g_tc_err);
        drain_bar(&bar_vfull[j % NS], (j / NS) & 1, &g_tc_err);
      }
    }
    __syncwarp();
    } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = ptx::idesc_bf16(128, 128, false, false);
      constexpr uint32_t IDESC_PV = ptx::idesc_bf16(128, D, false, true);
      const uint32_t aQ = ptx::smem_u32(sQ);
      const uint32_t aK = ptx::smem_u32(sK);
      const uint32_t aV = ptx::smem_u32(sV);
      bool ok = wait_bar(bar_q, 0, abort_flag, &g_tc_err, kErrWaitMma);
      ptx::tc_fence_after();

      // on an abort no further MMA is issued; those in flight are drained below
      auto issue_s = [&](int t, int j) -> bool {
        const int st = j % NS;
        if (!wait_bar(&bar_kfull[st], (j / NS) & 1, abort_flag, &g_tc_err, kErrWaitMma))
          return false;
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < Tile::QK_KSTEPS; ++kk)
          ptx::mma_ss(tmem + C::COL_S0 + t * 128, Tile::kmajor_desc(aQ + t * TILE, kk),
                      Tile::kmajor_desc(aK + st * TILE, kk), IDESC_QK, kk > 0 ? 1u : 0u);
        ptx::mma_commit(&bar_sfull[t]);
        return true;
      };

      if (ok && n_t0 > 0) ok = issue_s(0, 0);
      if (ok && n_t1 > 0) ok = issue_s(1, 0);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int st = j % NS;
        if (!wait_bar(&bar_vfull[st], (j / NS) & 1, abort_flag, &g_tc_err, kErrWaitMma)) break;
        ptx::tc_fence_after();
#pragma unroll 1
        for (int t = 0; t < 2; ++t) {
          const int nt = t == 0 ? n_t0 : n_t1;
          if (ok && j < nt) {
            // P arrives in chunks of 32 keys (two k-steps each): the tensor
            // core starts on the first chunk while the rest is computed
#pragma unroll
            for (int c = 0; c < C::P_CHUNKS; ++c) {
              if (!wait_bar(&bar_pfull[t * C::P_CHUNKS + c], j & 1, abort_flag, &g_tc_err,
                            kErrWaitMma)) {
                ok = false;
                break;
              }
              ptx::tc_fence_after();
              constexpr int KPC = Tile::PV_KSTEPS / C::P_CHUNKS;
#pragma unroll
              for (int kq = 0; kq < KPC; ++kq) {
                const int kk = c * KPC + kq;
                ptx::mma_ts(tmem + C::COL_O0 + t * 128, tmem + C::COL_S0 + t * 128 + kk * 8,
                            Tile::mnmajor_desc(aV + st * TILE, kk), IDESC_PV,
                            (j > 0 || kk > 0) ? 1u : 0u);
              }
            }
            if (!ok) break;
            ptx::mma_commit(&bar_odone[t]);
            const bool last_pv = (t == 1) || !(j < n_t1);
            if (last_pv) ptx::mma_commit(&bar_kvempty[st]);
            if (j + 1 < nt) ok = issue_s(t, j + 1);
          }
        }
      }
      ptx::mma_commit(bar_final);
      drain_bar(bar_final, 0, &g_tc_err);
    }
    __syncwarp();
    }
    teardown();
  } else {
    // ================================================ warpgroups 0, 1: softmax
    if constexpr (FA_TC_REG_SPLIT) ptx::setmaxnreg_inc<C::REGS_SOFTMAX>();
    const int t = warp >> 2;
    const int qr = warp & 3;
    const int row = qr * 32 + lane;
    const int q_start = q0 + 128 * t;
    const int grow = q_start + row;
    const uint32_t lane_off = static_cast<uint32_t>(qr * 32) << 16;
    const uint32_t tS = tmem + C::COL_S0 + t * 128 + lane_off;
    const uint32_t tO = tmem + C::COL_O0 + t * 128 + lane_off;
    const int n = t == 0 ? n_t0 : n_t1;
    const bool neg = scale_log2 < 0.f;
    const float mask_val = neg ? INFINITY : -INFINITY;
    float m_ref = -INFINITY;
    float l = 0.f;

    bool ok = true;
    for (int j = 0; j < n; ++j) {
      // warp-uniform decision: the tcgen05.ld/st below are warp-collective
      ok = __all_sync(0xffffffffu,
                      wait_bar(&bar_sfull[t], j & 1, abort_flag, &g_tc_err, kErrWaitSoftmax));
      if (!ok) break;
      ptx::tc_fence_after();
      uint32_t s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + c * 32, s[c]);
      ptx::tmem_ld_wait(s[0]);
      ptx::reg_fence(s[1]);
      ptx::reg_fence(s[2]);
      ptx::reg_fence(s[3]);

      // masked scores become -inf (+inf when scale < 0), so that their
      // scaled exponent is -inf and exp2 gives exactly 0 (scale_log2 is never
      // 0: the host passes the smallest normal float for scale = 0)
      const int kb = j * 128;
      const bool masked = (kb + 127 >= T) || (CAUSAL && kb + 127 > q_start);
      if (masked) {
        const int lim = CAUSAL ? min(T - 1, grow) - kb : T - 1 - kb;  // last kept column
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > lim) s[c >> 5][c & 31] = __float_as_uint(mask_val);
      }
      float mx;
      if (!neg) {
        float a0 = __uint_as_float(s[0][0]), a1 = __uint_as_float(s[1][0]);
        float a2 = __uint_as_float(s[2][0]), a3 = __uint_as_float(s[3][0]);
#pragma unroll
        for (int c = 1; c < 32; ++c) {
          a0 = fmaxf(a0, __uint_as_float(s[0][c]));
          a1 = fmaxf(a1, __uint_as_float(s[1][c]));
          a2 = fmaxf(a2, __uint_as_float(s[2][c]));
          a3 = fmaxf(a3, __uint_as_float(s[3][c]));
        }
        mx = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
      } else {
        float a0 = __uint_as_float(s[0][0]), a1 = __uint_as_float(s[1][0]);
        float a2 = __uint_as_float(s[2][0]), a3 = __uint_as_float(s[3][0]);
#pragma unroll
        for (int c = 1; c < 32; ++c) {
          a0 = fminf(a0, __uint_as_float(s[0][c]));
          a1 = fminf(a1, __uint_as_float(s[1][c]));
          a2 = fminf(a2, __uint_as_float(s[2][c]));
          a3 = fminf(a3, __uint_as_float(s[3][c]));
        }
        mx = fminf(fminf(a0, a1), fminf(a2, a3));
      }
      const float m_cand = mx * scale_log2;
      const bool resc = m_cand > m_ref + FA_RESCALE_THRESHOLD;
      float alpha = 1.f;
      if (resc) {
        alpha = ptx::ex2(m_ref - m_cand);  // 0 on the first tile (m_ref = -inf)
        m_ref = m_cand;
      }
      const float mo = (m_ref == -INFINITY) ? 0.f : m_ref;
      // the O correction comes first: the first P.V MMA of this tile
      // accumulates into O as soon as P chunk 0 is released
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
        if constexpr (D >= 32) {
#pragma unroll
          for (int oc = 0; oc < D / 32; ++oc) {
            uint32_t o[32];
            ptx::tmem_ld32(tO + oc * 32, o);
            ptx::tmem_ld_wait(o);
#pragma unroll
            for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
            ptx::tmem_st32(tO + oc * 32, o);
          }
        } else {
          uint32_t o[16];
          ptx::tmem_ld16(tO, o);
          ptx::tmem_ld_wait(o);
#pragma unroll
          for (int u = 0; u < 16; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
          ptx::tmem_st16(tO, o);
        }
      }
      float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float p0 = ptx::ex2(fmaf(__uint_as_float(s[c][2 * u]), scale_log2, -mo));
          const float p1 = ptx::ex2(fmaf(__uint_as_float(s[c][2 * u + 1]), scale_log2, -mo));
          sum0 += p0;
          sum1 += p1;
          pk[u] = ptx::pack_bf16x2(p0, p1);
        }
        ptx::tmem_st16(tS + c * 16, pk);
        // release a chunk of P once its keys are written: every lane's
        // stores are complete, then one lane per warp arrives (count 4)
        constexpr int PER = 4 / C::P_CHUNKS;  // 32-key pieces per chunk
        if ((c + 1) % PER == 0) {
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&bar_pfull[t * C::P_CHUNKS + c / PER]);
        }
      }
      l = l * alpha + (sum0 + sum1);
    }

    // ---- epilogue: O = O / l in bf16, L = m + ln l
    if (ok && n > 0)
      ok = __all_sync(0xffffffffu, wait_bar(&bar_odone[t], (n - 1) & 1, abort_flag, &g_tc_err,
                                            kErrWaitEpilogue));
    if (ok && n > 0) {
      ptx::tc_fence_after();
      const float inv_l = 1.f / l;
      const bool row_ok = grow < T;
      __nv_bfloat16* orow = O + (static_cast<size_t>(bh) * T + (row_ok ? grow : 0)) * D;
      if constexpr (D >= 32) {
#pragma unroll
        for (int oc = 0; oc < D / 32; ++oc) {
          uint32_t o[32];
          ptx::tmem_ld32(tO + oc * 32, o);
          ptx::tmem_ld_wait(o);
          uint32_t pk[16];
#pragma unroll
          for (int u = 0; u < 16; ++u)
            pk[u] = ptx::pack_bf16x2(__uint_as_float(o[2 * u]) * inv_l,
                                     __uint_as_float(o[2 * u + 1]) * inv_l);
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(orow + oc * 32);
#pragma unroll
            for (int w = 0; w < 4; ++w)
              dst[w] = make_uint4(pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
          }
        }
      } else {
        uint32_t o[16];
        ptx::tmem_ld16(tO, o);
        ptx::tmem_ld_wait(o);
        uint32_t pk[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          pk[u] = ptx::pack_bf16x2(__uint_as_float(o[2 * u]) * inv_l,
                                   __uint_as_float(o[2 * u + 1]) * inv_l);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow);
          dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
      if (row_ok)
        LSE[static_cast<size_t>(bh) * T + grow] = (m_ref + log2f(l)) * 0.6931471805599453f;
    }
    teardown();
  }
}

template <int D, bool CAUSAL>
static fa_status launch_tc_impl(const FwdArgs& a) {
  using C = TcCfg<D>;
  using Tile = TcTile<D>;
  auto kern = fa_fwd_tc_kernel<D, CAUSAL>;
  static bool attr_done = false;  // per instantiation; benign race (idempotent)
  if (!attr_done) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return cuda_status(e);
    // the register split must fit the launch allocation, else setmaxnreg.inc
    // would wait forever: refuse to launch instead
    cudaFuncAttributes fattr;
    e = cudaFuncGetAttributes(&fattr, kern);
    if (e != cudaSuccess) return cuda_status(e);
    if (C::REGS_SPLIT > C::THREADS * fattr.numRegs) return FA_ERR_UNSUPPORTED;
    attr_done = true;
  }
  CUtensorMap mq, mk, mv;
  CUresult r;
  if ((r = make_tmap_bf16(&mq, a.q, D, a.T, static_cast<long long>(a.B) * a.Hq, Tile::BOX_X,
                          Tile::TMA_SWIZZLE)) != CUDA_SUCCESS)
    return cu_status(r);
  if ((r = make_tmap_bf16(&mk, a.k, D, a.T, static_cast<long long>(a.B) * a.Hkv, Tile::BOX_X,
                          Tile::TMA_SWIZZLE)) != CUDA_SUCCESS)
    return cu_status(r);
  if ((r = make_tmap_bf16(&mv, a.v, D, a.T, static_cast<long long>(a.B) * a.Hkv, Tile::BOX_X,
                          Tile::TMA_SWIZZLE)) != CUDA_SUCCESS)
    return cu_status(r);
  const long long units = static_cast<long long>(a.B) * a.Hq * ((a.T + 255) / 256);
  // scale * log2(e); never exactly 0, so that masked (infinite) scores give
  // exponents of -inf rather than NaN: for scale = 0 the smallest normal
  // float stands in, and every finite score's exponent still rounds to 0
  float scale_log2 = a.scale * 1.4426950408889634f;
  if (scale_log2 == 0.f) scale_log2 = 1.17549435e-38f;
  kern<<<static_cast<unsigned>(units), C::THREADS, C::SMEM_BYTES, a.stream>>>(
      mq, mk, mv, static_cast<__nv_bfloat16*>(a.o), a.lse, a.B, a.Hq, a.Hkv, a.T, scale_log2);
  return cuda_status(cudaGetLastError());
}

fa_status launch_tc(const FwdArgs& a) {
  const bool c = a.causal != 0;
  switch (a.d) {
    case 16: return c ? launch_tc_impl<16, true>(a) : launch_tc_impl<16, false>(a);
    case 32: return c ? launch_tc_impl<32, true>(a) : launch_tc_impl<32, false>(a);
    case 64: return c ? launch_tc_impl<64, true>(a) : launch_tc_impl<64, false>(a);
    case 128: return c ? launch_tc_impl<128, true>(a) : launch_tc_impl<128, false>(a);
    default: return FA_ERR_UNSUPPORTED;
  }
}

fa_status tc_read_and_clear_error(unsigned int* word) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_err, sizeof(v));
  if (e != cudaSuccess) return cuda_status(e);
  if (v) {
    e = cudaMemcpyToSymbol(g_tc_err, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_status(e);
  }
  *word = v;
  return FA_OK;
}

}  // namespace fa
