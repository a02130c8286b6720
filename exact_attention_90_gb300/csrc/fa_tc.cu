// fa_tc.cu -- bf16 / fp16 exact attention forward on tcgen05 tensor cores (sm_103a).
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
// How it runs on Blackwell.  A work unit is 256 query rows of one (b, h), as
// two 128-row tiles Q0, Q1 that share every K/V tile loaded for them.  The
// grid is persistent: one CTA per SM walks the units in longest-first order,
// dealt in zig-zag rounds (forward, then backward) so the long causal units
// spread evenly; tensor memory and barriers are set up once, and the next
// unit's Q load and first S MMAs overlap the previous unit's epilogue.
// Warp roles:
//   warps 0-3 : softmax, correction and epilogue for Q0 (one thread per row)
//   warps 4-7 : the same for Q1
//   warp 8    : TMA producer (Q tiles through a ring of three slots, so
//               that the next unit's Q0 is loaded while this unit runs; K_j
//               and V_j through rings of NSK and NSV stages, released
//               separately)
//   warp 9    : MMA issuer for Q0
//   warp 10   : MMA issuer for Q1
//   (each issuer warp runs its loop on all 32 lanes, so that descriptors
//   and addresses stay warp-uniform values; one elected lane issues the
//   MMAs and commits)
//   warp 11 completes the third warpgroup, whose registers setmaxnreg hands
//   to the two softmax warpgroups
// Tensor memory (512 columns x 128 lanes x 32 bit), d = 128:
//   S0 [0,128)  S1 [128,256)  fp32 scores of Q0 K_j^T, Q1 K_j^T
//   P0, P1      bf16 probabilities packed two per column in the first 64
//               columns of S0 / S1 (written by the softmax warps)
//   O0 [256,256+d)  O1 [384,384+d)  fp32 output accumulators
// Per KV tile j the MMAs go out in the order PV0_j, S0_{j+1}, PV1_j, S1_{j+1};
// while the tensor core runs one tile's PV and next S, the other tile's
// softmax warps turn their S into P.  Each Q tile has its own issuer warp
// and the two hand a turn word back and forth, so that one issuer's waits and
// commits overlap the other's MMAs.  S_{t,j+1} overwrites the columns of
// P_{t,j}; it is issued after PV_{t,j} by the same thread (the issuer's
// elected lane), and tcgen05 MMAs of one thread execute in issue order.
// d <= 64 (SEP_P): the O accumulators take 2 x 64 columns, so P gets its own:
//   S0 [0,128)  S1 [128,256)  O0 [256,256+d)  O1 [320,320+d)
//   P0 [384,448)  P1 [448,512)
// and a tile's chain loses its MMA group: the softmax signals that it has
// read S_{t,j} (an S-read barrier), its issuer then computes S_{t,j+1} while
// the softmax is still exponentiating, and PV_{t,j} follows once P_{t,j} is
// stored.  The softmax stores P_{t,j} only after PV_{t,j-1} is done (the
// P.V-done barrier), which also orders its O correction.  The two issuers
// run without the turn word: their tiles share no tensor-memory columns.
// The softmax works in the log2 domain (scores times scale*log2(e), exp2 on
// the SFU) and rescales O lazily: the reference maximum is only raised when a
// row's maximum grows by more than 2^8, so most tiles skip the O correction;
// the result is exact because O and l always share the same reference.  At
// d <= 32 and d = 128 a tile after the row's first is exponentiated against
// the reference without its row maximum at all; the maximum, the rescale and
// the exponentials run again only when the tile's P sum reaches 2^15 (so no P
// can overflow fp16).
#include <cmath>
#include <cstdio>

#include "fa_internal.h"
#include "ptx.cuh"
#include "row_store.cuh"
#include "tc_layout.cuh"
#include "wait.cuh"

namespace fa {

static __device__ unsigned int g_tc_err;

// Tuning parameters (compile-time; defaults are the measured best):
//   FA_TC_REG_SPLIT  -- 1: 384 threads, setmaxnreg moves registers from the
//                       load/MMA warpgroup to the softmax warpgroups;
//                       0: 352 threads, one register budget for all warps
#ifndef FA_TC_REG_SPLIT
#define FA_TC_REG_SPLIT 1
#endif
//   FA_TC_K_STAGES_D128 -- depth of the K ring at d = 128 (2 or 3)
#ifndef FA_TC_K_STAGES_D128
#define FA_TC_K_STAGES_D128 2
#endif
//   FA_TC_ZIGZAG -- 1: units dealt forward on even rounds, backward on odd
//                   ones; 0: plain round robin
#ifndef FA_TC_ZIGZAG
#define FA_TC_ZIGZAG 1
#endif
//   FA_TC_PACKED_MATH -- 1: three-input max and paired fp32 FMA/add in the
//                        softmax (half the instructions); 0: scalar
#ifndef FA_TC_PACKED_MATH
#define FA_TC_PACKED_MATH 1
#endif

template <int D>
struct TcCfg : TcTile<D> {
  using Tile = TcTile<D>;
  // K and V ring depths.  K is free once both S MMAs of its tile are done,
  // V only after both P.V MMAs.  At d = 128: Q 3 x 32 KB + K 2 x 32 KB +
  // V 2 x 32 KB = 224 KB.
  static constexpr int NSK = D == 128 ? FA_TC_K_STAGES_D128 : 4;
  static constexpr int NSV = D == 128 ? 2 : 4;
  static constexpr int THREADS = FA_TC_REG_SPLIT ? 384 : 352;  // softmax Q0, Q1; load/MMA
  static constexpr int REGS_SOFTMAX = 200;  // per thread after setmaxnreg, warpgroups 0 and 1
  static constexpr int REGS_OTHER = 88;     // warpgroup 2
  // registers the three warpgroups hold after reallocation
  static constexpr int REGS_SPLIT = FA_TC_REG_SPLIT ? 128 * (2 * REGS_SOFTMAX + REGS_OTHER) : 0;
  static constexpr int NQ = 3;  // Q tile slots: a unit's Q0, Q1 and the next unit's Q0
  static constexpr int SMEM_BYTES = 1024 + (NQ + NSK + NSV) * Tile::TILE_BYTES + 512;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA exceeded");
  // the 512 bytes after the tiles: the barriers, the TMEM address, the abort
  // flag and the issue-turn word
  static_assert((2 * NQ + 2 * NSK + 2 * NSV + 9) * 8 + 3 * 4 <= 512, "barrier area exceeded");
  static constexpr uint32_t TMEM_COLS = 512;
  // SEP_P (d <= 64): P of tile t has its own 64 columns at COL_P0 + 64 t
  // instead of the first 64 columns of S_t, so that S_t(j+1) may be issued
  // as soon as the softmax has read S_t(j); at d = 128 the O accumulators
  // take those columns and P overwrites S.
  static constexpr bool SEP_P = D <= 64;
  static constexpr uint32_t COL_S0 = 0, COL_O0 = 256;
  static constexpr uint32_t O_STRIDE = SEP_P ? 64 : 128;  // O_t at COL_O0 + O_STRIDE t
  static constexpr uint32_t COL_P0 = SEP_P ? 384 : COL_S0;
  static constexpr uint32_t P_STRIDE = SEP_P ? 64 : 128;  // P_t at COL_P0 + P_STRIDE t
  // SPEC_EXP (d <= 32 and d = 128): exponentials against the running
  // reference without the row maximum (see the softmax).  A redo reads S
  // again from tensor memory, so S must stay there until the decision: at
  // d <= 32 the S-read signal waits for the exponentials, at d = 128 the
  // first half of P is stored early only on the redo path.  At d = 64 the
  // later S-read signal delays the next S (four MMA k-steps) by more than
  // the maximum saves.
  static constexpr bool SPEC_EXP = (SEP_P && D <= 32) || D == 128;
};

// log2 headroom of the lazy rescale: P values stay below 2^8
#define FA_RESCALE_THRESHOLD 8.0f

// KV tiles [lo, hi) that the 128 query rows starting at qs need: the keys
// [qs - wl, qs + 127 + wr] of the band mask (wl or wr < 0: unbounded side)
// inside [0, T); no mask is (-1, -1), causal attention (-1, 0).  Empty
// (lo = hi = 0) for rows past T.
__host__ __device__ __forceinline__ void tc_tile_range(int qs, int T, int wl, int wr, int& lo,
                                                       int& hi) {
  if (qs >= T) {
    lo = hi = 0;
    return;
  }
  lo = wl < 0 ? 0 : max(0, qs - wl) >> 7;
  const long long last =
      wr < 0 ? static_cast<long long>(T) - 1
             : min(static_cast<long long>(T) - 1, static_cast<long long>(qs) + 127 + wr);
  hi = static_cast<int>(last >> 7) + 1;
}

// One work unit: 256 query rows [q0, q0 + 256) of (b, h) as two 128-row
// tiles, over the KV tiles [j0, j0 + cnt) of split sp (of S).  Q tile t visits
// the local tiles [s_t, e_t) of them (s_t = e_t = 0: none); cnt = 0 marks an
// empty split, which every role skips.  The two intervals overlap or touch
// (a band keeps at least the diagonal key of every row), so every local tile
// is visited by at least one Q tile.
struct TcUnit {
  int bh, b, hk, q0, sp, j0, s0, e0, s1, e1, cnt;
  // local-global masks: the unit's KV tiles are the nb global tiles below
  // its band, the nband band tiles from j0 on, then the global tiles from
  // list index ia on (below, j0 + j is the band's tile for nb = 0); with
  // packed global keys: nb = 0, the band tiles, then np packed tiles
  int nb, nband, ia, np;
};

__device__ __forceinline__ TcUnit tc_unit(int idx, int B, int Hq, int Hkv, int T, int S, int wl,
                                          int wr) {
  TcUnit u;
  const int BH = B * Hq;
  const int n_qb = (T + 255) >> 8;
  u.sp = idx % S;
  const int rest = idx / S;
  const int qb = n_qb - 1 - rest / BH;  // last (longest when causal) row blocks first
  u.bh = rest % BH;
  u.b = u.bh / Hq;
  const int h = u.bh - u.b * Hq;
  u.hk = h / (Hq / Hkv);
  u.q0 = qb * 256;
  int lo0, hi0, lo1, hi1;
  tc_tile_range(u.q0, T, wl, wr, lo0, hi0);
  tc_tile_range(u.q0 + 128, T, wl, wr, lo1, hi1);
  int ulo = lo0, uhi = hi0;
  if (hi1 > lo1) {
    ulo = min(ulo, lo1);
    uhi = max(uhi, hi1);
  }
  const int chunk = (uhi - ulo + S - 1) / S;  // KV tiles per split of this row block
  u.j0 = ulo + u.sp * chunk;
  const int j1 = min(uhi, u.j0 + chunk);
  u.cnt = max(0, j1 - u.j0);
  // with no left bound every row's keys start at key 0, so both tiles start
  // at the split's first tile
  u.s0 = wl < 0 ? 0 : max(0, lo0 - u.j0);
  u.e0 = min(u.cnt, hi0 - u.j0);
  if (u.e0 <= u.s0) u.s0 = u.e0 = 0;
  u.s1 = wl < 0 ? 0 : max(0, lo1 - u.j0);
  u.e1 = min(u.cnt, hi1 - u.j0);
  if (u.e1 <= u.s1) u.s1 = u.e1 = 0;
  u.nb = 0;
  u.nband = u.cnt;
  u.ia = 0;
  u.np = 0;
  return u;
}

// a bounded barrier wait by every lane of a warp, with a warp-uniform result
__device__ __forceinline__ bool tc_wait_all(uint64_t* bar, uint32_t parity,
                                            volatile int* abort_flag, unsigned int* err,
                                            unsigned int code) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, err, code));
}

// first index of the sorted list[0, n) whose entry is >= x (n if none)
__device__ __forceinline__ int tc_lower_bound(const int* list, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(list + mid) < x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// A unit of the local-global mask (no KV split): the union of both Q tiles'
// bands [ulo, uhi) plus every tile holding a global key below ulo, or from
// uhi up to the last tile any row of the unit may see (its own last row's
// tile when causal).  Both Q tiles visit every tile of the unit; the mask
// removes what a row does not see.
//
// With packed global keys (`packed`: the sorted distinct tokens gtok[0,
// *gntok) in 128-row packed K/V tiles) the unit visits its band tiles and
// then every packed tile holding a token its rows may see (up to its last
// row when causal): a global key costs a packed row, not a whole tile.
__device__ __forceinline__ TcUnit tc_unit_lg(int idx, int B, int Hq, int Hkv, int T, int wl,
                                             int wr, int causal, const int* glist,
                                             const int* gcount, int packed, const int* gtok,
                                             const int* gntok) {
  TcUnit u = tc_unit(idx, B, Hq, Hkv, T, 1, wl, wr);
  if (packed) {
    const int G = __ldg(gntok);
    const int g_hi = causal ? tc_lower_bound(gtok, G, min(T - 1, u.q0 + 255) + 1) : G;
    u.nband = u.cnt;
    u.np = (g_hi + 127) >> 7;
    u.cnt = u.nband + u.np;
    u.s0 = u.s1 = 0;
    u.e0 = u.q0 < T ? u.cnt : 0;
    u.e1 = u.q0 + 128 < T ? u.cnt : 0;
    return u;
  }
  const int ulo = u.j0, uhi = u.j0 + u.cnt;
  const int n = __ldg(gcount);
  const int cap = causal ? min(T - 1, u.q0 + 255) >> 7 : (T - 1) >> 7;
  u.nb = tc_lower_bound(glist, n, ulo);
  u.ia = tc_lower_bound(glist, n, uhi);
  const int na = max(0, tc_lower_bound(glist, n, cap + 1) - u.ia);
  u.nband = u.cnt;
  u.cnt = u.nb + u.nband + na;
  u.s0 = u.s1 = 0;
  u.e0 = u.q0 < T ? u.cnt : 0;
  u.e1 = u.q0 + 128 < T ? u.cnt : 0;
  return u;
}

// Bits e of a 32-column group starting at column `base` with lo <= base + e <= hi.
__device__ __forceinline__ uint32_t tc_range_bits(int lo, int hi, int base) {
  const int a = max(lo - base, 0), b = min(hi - base, 31);
  if (a > b) return 0u;
  const uint32_t upto_b = b >= 31 ? 0xffffffffu : ((1u << (b + 1)) - 1u);
  const uint32_t below_a = (1u << a) - 1u;  // a <= 31 here
  return upto_b & ~below_a;
}

// KV tile of the unit's j-th visited tile
template <bool LG>
__device__ __forceinline__ int tc_tile_of(const TcUnit& u, int j, const int* glist) {
  if constexpr (!LG) {
    return u.j0 + j;
  } else {
    if (j < u.nb) return __ldg(glist + j);
    if (j < u.nb + u.nband) return u.j0 + (j - u.nb);
    return __ldg(glist + u.ia + (j - u.nb - u.nband));
  }
}

// The k-th unit of this CTA: rounds of gridDim.x units, dealt forward on even
// rounds and backward on odd ones.
__device__ __forceinline__ int tc_unit_index(int k) {
  const int G = static_cast<int>(gridDim.x), bid = static_cast<int>(blockIdx.x);
  return k * G + ((FA_TC_ZIGZAG && (k & 1)) ? G - 1 - bid : bid);
}

// Mask kinds, fixed at compile time so that the unmasked and causal kernels
// carry no window arithmetic: no mask, causal (j <= i), or a band given by
// the kernel's window arguments
enum : int { kMaskNone = 0, kMaskCausal = 1, kMaskBand = 2, kMaskLocalGlobal = 3 };

// F16: fp16 operands and output (else bf16); accumulation is fp32 either way
template <int D, int MASK, bool F16>
__global__ void __launch_bounds__(FA_TC_REG_SPLIT ? 384 : 352, 1)
    fa_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, uint16_t* __restrict__ O,
                     float* __restrict__ LSE, int B, int Hq, int Hkv, int T, float scale_log2,
                     int num_units, int S, float* __restrict__ part_o,
                     float* __restrict__ part_lse, int window_left, int window_right,
                     const uint32_t* __restrict__ lg_bits, const int* __restrict__ lg_list,
                     const int* __restrict__ lg_count, int lg_causal,
                     const __grid_constant__ CUtensorMap tmKg,
                     const __grid_constant__ CUtensorMap tmVg, int lg_packed,
                     const int* __restrict__ lg_tokens, const int* __restrict__ lg_ntok) {
  constexpr bool LG = MASK == kMaskLocalGlobal;
  // the band [i - wl, i + wr] of the mask kind (a negative side: unbounded)
  const int wl = (MASK == kMaskBand || LG) ? window_left : -1;
  const int wr = (MASK == kMaskBand || LG) ? window_right : (MASK == kMaskCausal ? 0 : -1);
  auto unit_at = [&](int idx) {
    if constexpr (LG)
      return tc_unit_lg(idx, B, Hq, Hkv, T, wl, wr, lg_causal, lg_list, lg_count, lg_packed,
                        lg_tokens, lg_ntok);
    else return tc_unit(idx, B, Hq, Hkv, T, S, wl, wr);
  };
  using C = TcCfg<D>;
  using Tile = TcTile<D>;
  constexpr int NSK = C::NSK, NSV = C::NSV;
  constexpr int TILE = Tile::TILE_BYTES;

  extern __shared__ uint8_t smem_raw[];
  // Shared-memory carve-up, recomputed where it is used: values computed
  // before the per-warpgroup register reallocation would have to survive
  // it (ptxas spills them), while these few integer operations are free.
  struct Smem {
    uint8_t *sQ, *sK, *sV;
    uint64_t *qfull, *qempty, *kfull, *vfull, *kempty, *vempty, *sfull, *pfull, *odone, *sread,
        *final_;
    uint32_t* tmem_slot;
    volatile int* abort_flag;
    volatile int* turn;  // MMA issue turn of the two issuing threads
    __device__ __forceinline__ explicit Smem(uint8_t* raw) {
      uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
      sQ = sm;                  // NQ Q tile slots
      sK = sm + C::NQ * TILE;   // NSK K tiles
      sV = sK + NSK * TILE;     // NSV V tiles
      uint64_t* bars = reinterpret_cast<uint64_t*>(sV + NSV * TILE);
      qfull = bars;             // [NQ] Q tile of the slot loaded
      qempty = bars + C::NQ;    // [NQ] the tile's last S MMA is done
      kfull = bars + 2 * C::NQ;
      vfull = kfull + NSK;
      kempty = vfull + NSV;     // K stage free: both issuers are past its S MMAs
      vempty = kempty + NSK;    // V stage free: both issuers are past its P.V MMAs
      sfull = vempty + NSV;     // [2]
      pfull = sfull + 2;        // [2]
      odone = pfull + 2;        // [2] the tile's last P.V done (SEP_P: every P.V)
      sread = odone + 2;        // [2] SEP_P: the softmax has read the tile's S
      final_ = sread + 2;
      tmem_slot = reinterpret_cast<uint32_t*>(final_ + 1);
      abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
      turn = abort_flag + 1;
    }
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // a programmatic dependent of this grid (the split merge) may be scheduled
  // from now on; it waits for this grid's completion before it reads
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) {
    const Smem m(smem_raw);
    uint64_t *bar_qfull = m.qfull, *bar_qempty = m.qempty, *bar_kfull = m.kfull,
             *bar_kempty = m.kempty, *bar_vfull = m.vfull, *bar_vempty = m.vempty,
             *bar_sfull = m.sfull, *bar_pfull = m.pfull, *bar_odone = m.odone,
             *bar_final = m.final_;
    volatile int* abort_flag = m.abort_flag;
    // the release barriers take one commit from each of the two MMA issuers
    for (int s = 0; s < C::NQ; ++s) {
      ptx::mbar_init(&bar_qfull[s], 1);
      ptx::mbar_init(&bar_qempty[s], 1);  // only the tile's own issuer reads it
    }
    for (int s = 0; s < NSK; ++s) {
      ptx::mbar_init(&bar_kfull[s], 1);
      ptx::mbar_init(&bar_kempty[s], 2);
    }
    for (int s = 0; s < NSV; ++s) {
      ptx::mbar_init(&bar_vfull[s], 1);
      ptx::mbar_init(&bar_vempty[s], 2);
    }
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(&bar_sfull[t], 1);
      ptx::mbar_init(&bar_pfull[t], 4);  // one elected lane per softmax warp
      ptx::mbar_init(&bar_odone[t], 1);
      ptx::mbar_init(&m.sread[t], 4);  // one elected lane per softmax warp
    }
    ptx::mbar_init(bar_final, 2);
    *abort_flag = 0;
    *m.turn = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(Smem(smem_raw).tmem_slot, C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();

  // every role ends here: all tensor-memory traffic is done before warp 0
  // frees the columns
  auto teardown = [&](uint32_t tmem) {
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
    const Smem m(smem_raw);
    uint8_t *sQ = m.sQ, *sK = m.sK, *sV = m.sV;
    uint64_t *bar_qfull = m.qfull, *bar_qempty = m.qempty, *bar_kfull = m.kfull,
             *bar_kempty = m.kempty, *bar_vfull = m.vfull, *bar_vempty = m.vempty,
             *bar_sfull = m.sfull, *bar_pfull = m.pfull, *bar_odone = m.odone,
             *bar_final = m.final_;
    volatile int* abort_flag = m.abort_flag;
    const uint32_t tmem = *m.tmem_slot;
    if (warp == 8) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        ptx::prefetch_tmap(&tmQ);
        ptx::prefetch_tmap(&tmK);
        ptx::prefetch_tmap(&tmV);
        const uint64_t pol_kv = ptx::policy_evict_last();
        const uint64_t pol_q = ptx::policy_evict_first();
        int q_issued = 0, kc = 0, vc = 0;  // Q, K, V tiles loaded so far
        bool ok = true;
        for (int k = 0; ok; ++k) {
          const int idx = tc_unit_index(k);
          if (idx >= num_units) break;
          const TcUnit u = unit_at(idx);
          if (u.cnt == 0) continue;
          // Q tile i (Q0, Q1 of each unit in turn) goes to slot i % NQ once
          // the tile NQ before it has had its last S MMA.  With three slots
          // the next unit's Q0 loads while this unit still runs; its Q1,
          // which takes this unit's Q0 slot, follows the first K and V tiles
          auto load_q = [&](int t) -> bool {
            const int sq = q_issued % C::NQ;
            if (q_issued >= C::NQ && !wait_bar(&bar_qempty[sq], ((q_issued / C::NQ) - 1) & 1,
                                               abort_flag, &g_tc_err, kErrWaitLoad))
              return false;
            ptx::mbar_arrive_expect_tx(&bar_qfull[sq], TILE);
#pragma unroll
            for (int bx = 0; bx < Tile::NBOX; ++bx)
              ptx::tma_load_3d_hint(sQ + sq * TILE + bx * Tile::BOX_BYTES, &tmQ, &bar_qfull[sq],
                                    bx * 64, u.q0 + 128 * t, u.bh, pol_q);
            ++q_issued;
            return true;
          };
          if (!load_q(0)) break;
          const int zkv = u.b * Hkv + u.hk;
          // KV tile of the unit's jj-th visited tile: a packed tile of global
          // keys (local-global) or a KV tile
          auto load_k = [&](int jj) -> bool {
            const bool pk = LG && lg_packed && jj >= u.nband;
            const int j = pk ? jj - u.nband : tc_tile_of<LG>(u, jj, lg_list);
            const int sk = kc % NSK;
            if (kc >= NSK && !wait_bar(&bar_kempty[sk], ((kc / NSK) - 1) & 1, abort_flag,
                                       &g_tc_err, kErrWaitLoad))
              return false;
            ptx::mbar_arrive_expect_tx(&bar_kfull[sk], TILE);
#pragma unroll
            for (int bx = 0; bx < Tile::NBOX; ++bx)
              ptx::tma_load_3d_hint(sK + sk * TILE + bx * Tile::BOX_BYTES, pk ? &tmKg : &tmK,
                                    &bar_kfull[sk], bx * 64, j * 128, zkv, pol_kv);
            ++kc;
            return true;
          };
          auto load_v = [&](int jj) -> bool {
            const bool pk = LG && lg_packed && jj >= u.nband;
            const int j = pk ? jj - u.nband : tc_tile_of<LG>(u, jj, lg_list);
            const int sv = vc % NSV;
            if (vc >= NSV && !wait_bar(&bar_vempty[sv], ((vc / NSV) - 1) & 1, abort_flag,
                                       &g_tc_err, kErrWaitLoad))
              return false;
            ptx::mbar_arrive_expect_tx(&bar_vfull[sv], TILE);
#pragma unroll
            for (int bx = 0; bx < Tile::NBOX; ++bx)
              ptx::tma_load_3d_hint(sV + sv * TILE + bx * Tile::BOX_BYTES, pk ? &tmVg : &tmV,
                                    &bar_vfull[sv], bx * 64, j * 128, zkv, pol_kv);
            ++vc;
            return true;
          };
          if constexpr (C::SEP_P) {
            // the issuers need K_{j+1} (the next S) before V_j (this P.V):
            // K runs one tile ahead of V
            for (int jj = 0; jj <= u.cnt; ++jj) {
              if ((jj < u.cnt && !load_k(jj)) || (jj == 0 && !load_q(1)) ||
                  (jj >= 1 && !load_v(jj - 1))) {
                ok = false;
                break;
              }
            }
          } else {
            for (int jj = 0; jj < u.cnt; ++jj) {
              if (!load_k(jj) || !load_v(jj) || (jj == 0 && !load_q(1))) {
                ok = false;
                break;
              }
            }
          }
        }
        // own copies still in flight (only after an abort) land before exit
        for (int c = max(0, q_issued - C::NQ); c < q_issued; ++c)
          drain_bar(&bar_qfull[c % C::NQ], (c / C::NQ) & 1, &g_tc_err);
        for (int c = max(0, kc - NSK); c < kc; ++c)
          drain_bar(&bar_kfull[c % NSK], (c / NSK) & 1, &g_tc_err);
        for (int c = max(0, vc - NSV); c < vc; ++c)
          drain_bar(&bar_vfull[c % NSV], (c / NSV) & 1, &g_tc_err);
      }
      __syncwarp();
    } else if (warp == 9 || warp == 10) {
      // ---------------------------------------------------------- MMA issuers
      // One issuer per Q tile (warp 9: Q0, warp 10: Q1).  The MMA groups keep
      // the order PV0_j S0_{j+1} | PV1_j S1_{j+1} | PV0_{j+1} ... through a
      // turn word: a thread waits for its P tile and its loads first, takes
      // its turn, issues its group, passes the turn, and only then commits
      // the S and K releases, so its commits and waits overlap the other
      // thread's MMAs (the V release goes between the group's P.V and S).  (Two
      // independent issuers let the tiles fall into step and their softmax
      // warpgroups contend; the alternation keeps them half a step apart.)
      // The whole warp runs the issue loop (every branch below is warp-
      // uniform: waits and the turn end in a vote); one elected lane issues
      // the MMAs and commits.  With the loop in lane 0 alone the operands
      // were not warp-uniform values and each MMA issued more slowly.
      {
        const int t = warp - 9;
        constexpr uint32_t IDESC_QK = ptx::idesc_16bit(128, 128, false, false, F16);
        constexpr uint32_t IDESC_PV = ptx::idesc_16bit(128, D, false, true, F16);
        const uint32_t aQ = ptx::smem_u32(sQ);
        const uint32_t aK = ptx::smem_u32(sK);
        const uint32_t aV = ptx::smem_u32(sV);
        volatile int* turn = m.turn;
        int kc = 0, vc = 0;  // K, V tiles consumed so far
        int pc = 0;          // P tiles of this Q tile consumed so far
        int nu = 0;          // units processed so far
        int ng = 0;          // turns taken so far
        bool ok = true;
        // bounded wait for this thread's turn (2 ng + t)
        auto take_turn = [&]() -> bool {
          const int want = 2 * ng + t;
          if (*turn == want) return true;
          const long long t0 = clock64();
          while (*turn != want) {
            if (*abort_flag) return false;
            if (clock64() - t0 > FA_WAIT_BUDGET_CYCLES) {
              *abort_flag = 1;
              atomicOr(&g_tc_err, kErrWaitMma);
              return false;
            }
          }
          return true;
        };
        auto pass_turn = [&]() {
          *turn = 2 * ng + t + 1;
          ++ng;
        };
        if constexpr (C::SEP_P) {
        // Separate P columns: this thread issues S_t(j+1) as soon as the
        // softmax has read S_t(j) and P.V_t(j) once P_t(j) is ready, without
        // a turn; the other tile's thread does the same for its tile.  Its
        // own MMAs execute in issue order, and the two tiles share no
        // tensor-memory columns.
        int sc = 0;  // S tiles issued (phases of this tile's S-read barrier)
        for (int k = 0; ok; ++k) {
          const int idx = tc_unit_index(k);
          if (idx >= num_units) break;
          const TcUnit u = unit_at(idx);
          if (u.cnt == 0) continue;
          const int sq = (2 * nu + t) % C::NQ;
          if (!tc_wait_all(&bar_qfull[sq], ((2 * nu + t) / C::NQ) & 1, abort_flag, &g_tc_err,
                        kErrWaitMma))
            break;
          ++nu;
          const uint32_t qlo = Tile::kmajor_lo(aQ + sq * TILE);
          ptx::tc_fence_after();
          const int js = t == 0 ? u.s0 : u.s1;
          const int je = t == 0 ? u.e0 : u.e1;
          for (int j = -1; ok && j < u.cnt; ++j) {
            const bool pv = j >= 0 && j >= js && j < je;
            const bool sn = j + 1 < u.cnt && j + 1 >= js && j + 1 < je;
            const int cv = vc + j, ck = kc + j + 1;
            if (j + 1 < u.cnt) {
              // both threads wait for every load before releasing its stage
              if (!tc_wait_all(&bar_kfull[ck % NSK], (ck / NSK) & 1, abort_flag, &g_tc_err,
                               kErrWaitMma)) {
                ok = false;
                break;
              }
              if (sn) {
                if (sc > 0 && !tc_wait_all(&m.sread[t], (sc - 1) & 1, abort_flag, &g_tc_err,
                                           kErrWaitMma)) {
                  ok = false;
                  break;
                }
                ptx::tc_fence_after();
                const uint32_t klo = Tile::kmajor_lo(aK + (ck % NSK) * TILE);
#pragma unroll
                for (int kk = 0; kk < Tile::QK_KSTEPS; ++kk)
                  ptx::mma_ss_lh_e(tmem + C::COL_S0 + t * 128, qlo + Tile::kmajor_step(kk),
                                   Tile::DESC_HI, klo + Tile::kmajor_step(kk), Tile::DESC_HI,
                                   IDESC_QK, kk > 0 ? 1u : 0u);
                ptx::mma_commit_e(&bar_sfull[t]);
                ++sc;
              }
              ptx::mma_commit_e(&bar_kempty[ck % NSK]);
            }
            // Q is free once this thread's last S of the unit is issued
            if (j + 1 == (je > js ? je - 1 : 0)) ptx::mma_commit_e(&bar_qempty[sq]);
            if (j >= 0) {
              if (!tc_wait_all(&bar_vfull[cv % NSV], (cv / NSV) & 1, abort_flag, &g_tc_err,
                               kErrWaitMma)) {
                ok = false;
                break;
              }
              if (pv) {
                if (!tc_wait_all(&bar_pfull[t], pc & 1, abort_flag, &g_tc_err, kErrWaitMma)) {
                  ok = false;
                  break;
                }
                ++pc;
                ptx::tc_fence_after();
                const uint32_t vlo = Tile::mnmajor_lo(aV + (cv % NSV) * TILE);
#pragma unroll
                for (int kk = 0; kk < Tile::PV_KSTEPS; ++kk)
                  ptx::mma_ts_lh_e(tmem + C::COL_O0 + t * C::O_STRIDE,
                                   tmem + C::COL_P0 + t * C::P_STRIDE + kk * 8,
                                   vlo + Tile::mnmajor_step(kk), Tile::DESC_HI, IDESC_PV,
                                   (j > js || kk > 0) ? 1u : 0u);
                ptx::mma_commit_e(&bar_odone[t]);  // P_t and O_t free again
              }
              ptx::mma_commit_e(&bar_vempty[cv % NSV]);
            }
          }
          kc += u.cnt;
          vc += u.cnt;
        }
        } else {
        for (int k = 0; ok; ++k) {
          const int idx = tc_unit_index(k);
          if (idx >= num_units) break;
          const TcUnit u = unit_at(idx);
          if (u.cnt == 0) continue;
          // this thread's Q tile of the unit: tile 2 nu + t of the Q ring
          const int sq = (2 * nu + t) % C::NQ;
          if (!tc_wait_all(&bar_qfull[sq], ((2 * nu + t) / C::NQ) & 1, abort_flag, &g_tc_err,
                        kErrWaitMma))
            break;
          ++nu;
          const uint32_t qlo = Tile::kmajor_lo(aQ + sq * TILE);
          ptx::tc_fence_after();
          const int js = t == 0 ? u.s0 : u.s1;
          const int je = t == 0 ? u.e0 : u.e1;
          // one turn per step: [P.V_t(j) when this tile visits KV tile j]
          // [S_t(j+1) when it visits j+1]; step -1 holds only S_t(0)
          for (int j = -1; ok && j < u.cnt; ++j) {
            const bool pv = j >= 0 && j >= js && j < je;
            const bool sn = j + 1 < u.cnt && j + 1 >= js && j + 1 < je;
            const int cv = vc + j, ck = kc + j + 1;
            // the loads are waited for by both threads even when the tile is
            // not theirs: a release commit before the load has landed would
            // count towards the stage's previous phase
            if (j >= 0 && !tc_wait_all(&bar_vfull[cv % NSV], (cv / NSV) & 1, abort_flag, &g_tc_err,
                                    kErrWaitMma)) {
              ok = false;
              break;
            }
            if (j + 1 < u.cnt && !tc_wait_all(&bar_kfull[ck % NSK], (ck / NSK) & 1, abort_flag,
                                           &g_tc_err, kErrWaitMma)) {
              ok = false;
              break;
            }
            if (pv && !tc_wait_all(&bar_pfull[t], pc & 1, abort_flag, &g_tc_err, kErrWaitMma)) {
              ok = false;
              break;
            }
            if (!__all_sync(0xffffffffu, take_turn())) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            if (pv) {
              ++pc;
              const uint32_t vlo = Tile::mnmajor_lo(aV + (cv % NSV) * TILE);
#pragma unroll
              for (int kk = 0; kk < Tile::PV_KSTEPS; ++kk)
                ptx::mma_ts_lh_e(tmem + C::COL_O0 + t * C::O_STRIDE,
                                 tmem + C::COL_S0 + t * 128 + kk * 8,
                               vlo + Tile::mnmajor_step(kk), Tile::DESC_HI, IDESC_PV,
                               (j > js || kk > 0) ? 1u : 0u);
            }
            // V_j (and, after the tile's last P.V, O_t) are free once this
            // thread's P.V is done: committed before its next S, so that the
            // two-stage V ring reloads without waiting for that S as well
            if (pv && j == je - 1) ptx::mma_commit_e(&bar_odone[t]);
            if (j >= 0) ptx::mma_commit_e(&bar_vempty[cv % NSV]);
            if (sn) {
              const uint32_t klo = Tile::kmajor_lo(aK + (ck % NSK) * TILE);
#pragma unroll
              for (int kk = 0; kk < Tile::QK_KSTEPS; ++kk)
                ptx::mma_ss_lh_e(tmem + C::COL_S0 + t * 128, qlo + Tile::kmajor_step(kk),
                               Tile::DESC_HI, klo + Tile::kmajor_step(kk), Tile::DESC_HI,
                               IDESC_QK, kk > 0 ? 1u : 0u);
            }
            pass_turn();
            if (sn) ptx::mma_commit_e(&bar_sfull[t]);
            if (j + 1 < u.cnt) ptx::mma_commit_e(&bar_kempty[ck % NSK]);
            // Q is free once this thread's last S of the unit is issued
            if (j + 1 == (je > js ? je - 1 : 0)) ptx::mma_commit_e(&bar_qempty[sq]);
          }
          kc += u.cnt;
          vc += u.cnt;
        }
        }
        ptx::mma_commit_e(bar_final);
        drain_bar(bar_final, 0, &g_tc_err);
      }
      __syncwarp();
    }
    teardown(tmem);
  } else {
    // ================================================ warpgroups 0, 1: softmax
    if constexpr (FA_TC_REG_SPLIT) ptx::setmaxnreg_inc<C::REGS_SOFTMAX>();
    const Smem m(smem_raw);
    uint64_t *bar_sfull = m.sfull, *bar_pfull = m.pfull, *bar_odone = m.odone;
    volatile int* abort_flag = m.abort_flag;
    const uint32_t tmem = *m.tmem_slot;
    const int t = warp >> 2;
    const int qr = warp & 3;
    const int row = qr * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(qr * 32) << 16;
    const uint32_t tS = tmem + C::COL_S0 + t * 128 + lane_off;
    const uint32_t tO = tmem + C::COL_O0 + t * C::O_STRIDE + lane_off;
    const uint32_t tP = tmem + C::COL_P0 + t * C::P_STRIDE + lane_off;
    int pw = 0;  // SEP_P: P.V completions of this tile waited for
    const bool neg = scale_log2 < 0.f;
    const float mask_val = neg ? INFINITY : -INFINITY;
    int it = 0;  // S tiles of this Q tile processed so far (barrier phases)
    int ne = 0;  // epilogues of this Q tile so far (O-done phases)
    bool ok = true;

    for (int k = 0; ok; ++k) {
      const int idx = tc_unit_index(k);
      if (idx >= num_units) break;
      const TcUnit u = unit_at(idx);
      const int js = t == 0 ? u.s0 : u.s1;  // this Q tile's local KV tiles [js, je)
      const int je = t == 0 ? u.e0 : u.e1;
      const int n = je - js;
      const int q_start = u.q0 + 128 * t;
      const int grow = q_start + row;
      float m_ref = -INFINITY;
      float l = 0.f;
      // packed global keys: this row keeps packed positions [0, pk_c) outside
      // [pk_a, pk_b), the tokens in its band (the band tiles hold those) and,
      // when causal, those after the row excluded
      int pk_a = 0, pk_b = 0, pk_c = 0;
      if constexpr (LG) {
        if (lg_packed) {
          const int G = __ldg(lg_ntok);
          pk_a = wl < 0 ? 0 : tc_lower_bound(lg_tokens, G, grow - wl);
          pk_b = wr < 0 ? G : tc_lower_bound(lg_tokens, G, grow + wr + 1);
          pk_c = lg_causal ? tc_lower_bound(lg_tokens, G, grow + 1) : G;
        }
      }

      for (int j = js; j < je; ++j, ++it) {
        // warp-uniform decision: the tcgen05.ld/st below are warp-collective
        ok = __all_sync(0xffffffffu,
                        wait_bar(&bar_sfull[t], it & 1, abort_flag, &g_tc_err, kErrWaitSoftmax));
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t sflat[128];
        uint32_t(&s)[4][32] = *reinterpret_cast<uint32_t(*)[4][32]>(&sflat);
        // S of the tile into registers, masked
        auto load_s = [&]() {
          ptx::tmem_ld128(tS, sflat);
          ptx::tmem_ld_wait(sflat);

          // masked scores become -inf (+inf when scale < 0), so that their
          // scaled exponent is -inf and exp2 gives exactly 0 (scale_log2 is
          // never 0: the host passes the smallest normal float for scale = 0)
          // a tile needs the mask unless all its keys lie in every row's band
          // [row - wl, row + wr] and before T
          const bool pk = LG && lg_packed && j >= u.nband;  // a packed tile of global keys
          const int kb = pk ? 0 : tc_tile_of<LG>(u, j, lg_list) * 128;
          const bool inside = !pk && kb + 127 < T && (wr < 0 || kb + 127 <= q_start + wr) &&
                              (wl < 0 || kb >= q_start + 127 - wl);
          if (!inside && pk) {
            // packed positions [0, pk_c) outside [pk_a, pk_b), one keep word
            // per 32 columns
            const int pb = (j - u.nband) * 128;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const uint32_t keep = tc_range_bits(0, pk_c - 1 - pb, 32 * g) &
                                    ~tc_range_bits(pk_a - pb, pk_b - 1 - pb, 32 * g);
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (!((keep >> e) & 1u)) s[g][e] = __float_as_uint(mask_val);
            }
          } else if (!inside) {
            const int hi_c = (wr < 0 ? T - 1 : min(T - 1, grow + wr)) - kb;  // last kept column
            const int lo_c = wl < 0 ? -1 : grow - wl - kb;                     // first kept
            if constexpr (LG) {
              // band OR a global key (before T, and not after the row when
              // causal), as one keep word per 32 columns; with packed global
              // keys the band tiles keep their band only
              const uint4 g4 = lg_packed ? make_uint4(0u, 0u, 0u, 0u)
                                         : __ldg(reinterpret_cast<const uint4*>(lg_bits) +
                                                 (kb >> 7));
              const int ghi_c = (lg_causal ? min(T - 1, grow) : T - 1) - kb;
#pragma unroll
              for (int g = 0; g < 4; ++g) {
                const uint32_t gw = g == 0 ? g4.x : (g == 1 ? g4.y : (g == 2 ? g4.z : g4.w));
                const uint32_t keep = tc_range_bits(lo_c, hi_c, 32 * g) |
                                      (gw & tc_range_bits(0, ghi_c, 32 * g));
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  if (!((keep >> e) & 1u)) s[g][e] = __float_as_uint(mask_val);
              }
            } else {
              // the band's columns [lo_c, hi_c] as one keep word per 32 columns
#pragma unroll
              for (int g = 0; g < 4; ++g) {
                const uint32_t keep = tc_range_bits(lo_c, hi_c, 32 * g);
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  if (!((keep >> e) & 1u)) s[g][e] = __float_as_uint(mask_val);
              }
            }
          }
        };
        load_s();
        auto signal_s_read = [&]() {
          if constexpr (C::SEP_P) {
            // S_t(j) is no longer needed: the issuer may compute S_t(j+1) into it
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&m.sread[t]);
          }
        };
        if constexpr (!C::SPEC_EXP) signal_s_read();
        // P = 2^(s * scale_log2 - m) for two keys at a time (paired FMA),
        // rounded to bf16 pairs into the first 64 columns of S (d <= 64: into
        // P's own columns); l sums the unrounded values.  At d = 128 the first
        // 32 columns of P go to tensor memory while the second half is still
        // being computed, so that only half of the store is left after the
        // last exponential.
        const uint64_t sl2x2 = ptx::f2_pack(scale_log2, scale_log2);
        uint64_t acc2[2];
        uint32_t pall[64];
        bool early = false;  // d = 128: the first half of P already stored
        auto exps = [&](float mo, bool allow_early) {
          const uint64_t nmox2 = ptx::f2_pack(-mo, -mo);
          acc2[0] = acc2[1] = ptx::f2_pack(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if (D == 128 && allow_early && c == 2) {
              ptx::tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pall[0]));
              early = true;
            }
            uint32_t(&pk)[16] = *reinterpret_cast<uint32_t(*)[16]>(&pall[16 * c]);
#pragma unroll
            for (int v = 0; v < 16; ++v) {
              const uint64_t x2 = ptx::fma2(
                  ptx::f2_pack(__uint_as_float(s[c][2 * v]), __uint_as_float(s[c][2 * v + 1])),
                  sl2x2, nmox2);
              float x0, x1;
              ptx::f2_unpack(x2, x0, x1);
              const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
              acc2[v & 1] = ptx::add2(acc2[v & 1], ptx::f2_pack(p0, p1));
              pk[v] = ptx::pack_x2<F16>(p0, p1);
            }
          }
        };
        bool resc = false;
        float alpha = 1.f;
        bool slow = true;
        if constexpr (C::SPEC_EXP) {
          // After a row's first tile the exponentials run against the current
          // reference without the tile's row maximum: P may exceed the lazy
          // rescale's 2^8, which bf16/fp16 P and the fp32 sums absorb.  A
          // tile sum at or above 2^15 (or not finite) sends the warp through
          // the maximum, the rescale and the exponentials again, on S read
          // once more from tensor memory.
          slow = __any_sync(0xffffffffu, m_ref == -INFINITY);
          if (!slow) {
            exps(m_ref, false);
            const uint64_t t2 = ptx::add2(acc2[0], acc2[1]);
            float h0, h1;
            ptx::f2_unpack(t2, h0, h1);
            slow = __any_sync(0xffffffffu, !(h0 + h1 < 32768.f));
            if (slow) load_s();
          }
        }
        if (slow) {
          // row maximum (minimum when scale < 0) with four independent chains
          float a[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            a[c] = __uint_as_float(s[c][0]);
#pragma unroll
            for (int v = 1; v < 31; v += 2) {
              const float x = __uint_as_float(s[c][v]), y = __uint_as_float(s[c][v + 1]);
              a[c] = neg ? ptx::min3(a[c], x, y) : ptx::max3(a[c], x, y);
            }
          }
          float mx;
          if (!neg)
            mx = ptx::max3(ptx::max3(a[0], a[1], __uint_as_float(s[0][31])),
                           ptx::max3(a[2], a[3], __uint_as_float(s[1][31])),
                           fmaxf(__uint_as_float(s[2][31]), __uint_as_float(s[3][31])));
          else
            mx = ptx::min3(ptx::min3(a[0], a[1], __uint_as_float(s[0][31])),
                           ptx::min3(a[2], a[3], __uint_as_float(s[1][31])),
                           fminf(__uint_as_float(s[2][31]), __uint_as_float(s[3][31])));
          const float m_cand = mx * scale_log2;
          resc = m_cand > m_ref + FA_RESCALE_THRESHOLD;
          if (resc) {
            alpha = ptx::ex2(m_ref - m_cand);  // 0 on the first tile (m_ref = -inf)
            m_ref = m_cand;
          }
          exps((m_ref == -INFINITY) ? 0.f : m_ref, true);
        }
        if constexpr (C::SPEC_EXP) signal_s_read();
        if constexpr (C::SEP_P) {
          // P_t and O_t are free once P.V_t(j-1) is done (the unit's first
          // tile: the epilogue of the previous unit waited for its last)
          if (j > js) {
            ok = __all_sync(0xffffffffu, wait_bar(&bar_odone[t], (pw++) & 1, abort_flag,
                                                  &g_tc_err, kErrWaitSoftmax));
            if (!ok) break;
            ptx::tc_fence_after();
          }
          ptx::tmem_st64(tP, pall);
        } else if constexpr (D == 128) {
          if (early) ptx::tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pall[32]));
          else ptx::tmem_st64(tS, pall);
        } else {
          ptx::tmem_st64(tS, pall);
        }
        // O correction (lazy, warp-uniform), before P is released: the next
        // P.V MMA accumulates into O
        if (j > js && __any_sync(0xffffffffu, resc)) {
          if constexpr (D >= 32) {
#pragma unroll
            for (int oc = 0; oc < D / 32; ++oc) {
              uint32_t o[32];
              ptx::tmem_ld32(tO + oc * 32, o);
              ptx::tmem_ld_wait(o);
#pragma unroll
              for (int v = 0; v < 32; ++v) o[v] = __float_as_uint(__uint_as_float(o[v]) * alpha);
              ptx::tmem_st32(tO + oc * 32, o);
            }
          } else {
            uint32_t o[16];
            ptx::tmem_ld16(tO, o);
            ptx::tmem_ld_wait(o);
#pragma unroll
            for (int v = 0; v < 16; ++v) o[v] = __float_as_uint(__uint_as_float(o[v]) * alpha);
            ptx::tmem_st16(tO, o);
          }
        }
        // release P: every lane's stores are complete, then one lane per warp
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bar_pfull[t]);
        {
          const uint64_t t2 = ptx::add2(acc2[0], acc2[1]);
          float h0, h1;
          ptx::f2_unpack(t2, h0, h1);
          l = l * alpha + (h0 + h1);
        }
      }
      if (!ok || n == 0) continue;

      // ---- epilogue: O = O / l in bf16, L = m + ln l (the tensor core meanwhile
      // computes the next unit's first S tiles)
      ok = __all_sync(0xffffffffu, wait_bar(&bar_odone[t], (C::SEP_P ? pw++ : ne++) & 1,
                                            abort_flag, &g_tc_err,
                                            kErrWaitEpilogue));
      if (!ok) break;
      ptx::tc_fence_after();
      const float inv_l = 1.f / l;
      const bool row_ok = grow < T;
      if (part_o != nullptr) {
        // split of the KV range: normalised fp32 partial O and its LSE; the
        // combine kernel merges the splits
        const size_t prow = static_cast<size_t>(u.sp) * B * Hq * T +
                            static_cast<size_t>(u.bh) * T + (row_ok ? grow : 0);
        float* po = part_o + prow * D;
#pragma unroll
        for (int oc = 0; oc < (D + 31) / 32; ++oc) {
          uint32_t o[32];
          if constexpr (D >= 32) {
            ptx::tmem_ld32(tO + oc * 32, o);
            ptx::tmem_ld_wait(o);
          } else {
            uint32_t h16[16];
            ptx::tmem_ld16(tO, h16);
            ptx::tmem_ld_wait(h16);
#pragma unroll
            for (int v = 0; v < 16; ++v) o[v] = h16[v];
          }
          if (row_ok) {
            float4* dst = reinterpret_cast<float4*>(po + oc * 32);
#pragma unroll
            for (int w = 0; w < (D >= 32 ? 8 : 4); ++w)
              dst[w] = make_float4(__uint_as_float(o[4 * w]) * inv_l,
                                   __uint_as_float(o[4 * w + 1]) * inv_l,
                                   __uint_as_float(o[4 * w + 2]) * inv_l,
                                   __uint_as_float(o[4 * w + 3]) * inv_l);
          }
        }
        if (row_ok) part_lse[prow] = (m_ref + log2f(l)) * 0.6931471805599453f;
        ptx::tc_fence_before();
        continue;
      }
      // rows of the lane pair, written as whole 32-byte sectors (row_store.cuh)
      const RowPair rp = row_pair(O + static_cast<size_t>(u.bh) * T * D, D, grow, T, lane);
      if constexpr (D >= 32) {
#pragma unroll
        for (int oc = 0; oc < D / 32; ++oc) {
          uint32_t o[32];
          ptx::tmem_ld32(tO + oc * 32, o);
          ptx::tmem_ld_wait(o);
          uint32_t pk[16];
#pragma unroll
          for (int v = 0; v < 16; ++v)
            pk[v] = ptx::pack_x2<F16>(__uint_as_float(o[2 * v]) * inv_l,
                                      __uint_as_float(o[2 * v + 1]) * inv_l);
          store_sector_pair(rp, oc * 32, pk);
          store_sector_pair(rp, oc * 32 + 16, pk + 8);
        }
      } else {
        uint32_t o[16];
        ptx::tmem_ld16(tO, o);
        ptx::tmem_ld_wait(o);
        uint32_t pk[8];
#pragma unroll
        for (int v = 0; v < 8; ++v)
          pk[v] = ptx::pack_x2<F16>(__uint_as_float(o[2 * v]) * inv_l,
                                    __uint_as_float(o[2 * v + 1]) * inv_l);
        store_sector_pair(rp, 0, pk);
      }
      if (row_ok)
        LSE[static_cast<size_t>(u.bh) * T + grow] = (m_ref + log2f(l)) * 0.6931471805599453f;
      // the O reads above are complete before this warp releases its next P
      ptx::tc_fence_before();
    }
    teardown(tmem);
  }
}

// SMs of the current device (cached per device)
static int tc_sm_count() {
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

// Merge of the KV splits of one query row (one warp per row): with the
// splits' normalised partial outputs O_s and log-sum-exps L_s,
//   L = m + ln sum_s exp(L_s - m),  m = max_s L_s,
//   O = sum_s exp(L_s - L) O_s,
// the same online-softmax rescaling, applied across splits instead of tiles.
// Only the splits whose KV range reaches the row's tile are read.  The lanes
// read the splits' L_s side by side (32 at a time) and each lane owns four
// consecutive columns of O, so that the loads of all splits are independent
// of one another: the merge costs a few memory round trips, not two per
// split.  Launched as a programmatic dependent of the attention kernel: the
// grid may start early and waits here until that kernel's writes are visible.
template <bool F16>
__global__ void __launch_bounds__(256)
    fa_split_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                            uint16_t* __restrict__ O, float* __restrict__ LSE, int BH, int T,
                            int D, int S, int wl, int wr) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long rows = static_cast<long long>(BH) * T;
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int r = static_cast<int>(row % T);
  // the row's KV tiles, the unit's union of both Q tiles' ranges, and the
  // splits of that union (as the attention kernel cut them)
  const int q0 = (r >> 8) << 8;
  int lo0, hi0, lo1, hi1;
  tc_tile_range(q0, T, wl, wr, lo0, hi0);
  tc_tile_range(q0 + 128, T, wl, wr, lo1, hi1);
  int ulo = lo0, uhi = hi0;
  if (hi1 > lo1) {
    ulo = min(ulo, lo1);
    uhi = max(uhi, hi1);
  }
  const int chunk = (uhi - ulo + S - 1) / S;
  const bool second = ((r >> 7) & 1) != 0;
  const int rlo = second ? lo1 : lo0, rhi = second ? hi1 : hi0;
  // splits [ulo + sp * chunk, ...) that hold part of [rlo, rhi)
  const int sp_first = (rlo - ulo) / chunk;
  const int ns = min(S, (rhi - ulo + chunk - 1) / chunk);
  // four consecutive columns per lane (lanes past d re-read column 0 and
  // store nothing)
  const int c4 = lane * 4;
  const bool col_ok = c4 < D;
  const int c4c = col_ok ? c4 : 0;
  if (ns - sp_first <= 8) {
    // up to eight splits (the split heuristic's count): the partial-O loads
    // go out before the L_s loads and the weights, in the same memory round
    // trip, since they depend on neither
    const int cnt = ns - sp_first;
    float4 x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int sp = sp_first + min(u, cnt - 1);
      x[u] = __ldg(reinterpret_cast<const float4*>(part_o + (sp * rows + row) * D + c4c));
    }
    const float l_mine = lane < cnt ? part_lse[(sp_first + lane) * rows + row] : -INFINITY;
    float m8 = l_mine;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) m8 = fmaxf(m8, __shfl_xor_sync(0xffffffffu, m8, o));
    m8 = __shfl_sync(0xffffffffu, m8, 0);  // lanes 0-7 hold the splits
    const float w_mine = lane < cnt ? expf(l_mine - m8) : 0.f;
    float ws = w_mine;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
    ws = __shfl_sync(0xffffffffu, ws, 0);
    float4 a8 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float w = __shfl_sync(0xffffffffu, w_mine, u);  // 0 past the last split
      a8.x = fmaf(w, x[u].x, a8.x);
      a8.y = fmaf(w, x[u].y, a8.y);
      a8.z = fmaf(w, x[u].z, a8.z);
      a8.w = fmaf(w, x[u].w, a8.w);
    }
    const float inv8 = 1.f / ws;
    if (col_ok) {
      uint2 packed;
      packed.x = ptx::pack_x2<F16>(a8.x * inv8, a8.y * inv8);
      packed.y = ptx::pack_x2<F16>(a8.z * inv8, a8.w * inv8);
      *reinterpret_cast<uint2*>(O + row * D + c4) = packed;
    }
    if (lane == 0) LSE[row] = m8 + logf(ws);
    return;
  }
  // m = max_s L_s over the lanes' splits sp_first + lane + 32 i
  float m = -INFINITY;
  for (int sp = sp_first + lane; sp < ns; sp += 32) m = fmaxf(m, part_lse[sp * rows + row]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  // the weights of 32 splits at a time come from the lanes that read their
  // L_s.  Eight splits' loads are issued together, so that each batch costs
  // one memory round trip.
  float wsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int base = sp_first; base < ns; base += 32) {
    const int mine = base + lane;
    const float w_mine = mine < ns ? expf(part_lse[mine * rows + row] - m) : 0.f;
    wsum += w_mine;
    const int cnt = min(32, ns - base);
    for (int i0 = 0; i0 < cnt; i0 += 8) {
      float4 x[8];
      float w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = min(i0 + u, cnt - 1);  // past the last split: weight 0
        w[u] = __shfl_sync(0xffffffffu, w_mine, i);
        if (i0 + u >= cnt) w[u] = 0.f;
        x[u] = __ldg(reinterpret_cast<const float4*>(part_o + ((base + i) * rows + row) * D + c4c));
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        acc.x = fmaf(w[u], x[u].x, acc.x);
        acc.y = fmaf(w[u], x[u].y, acc.y);
        acc.z = fmaf(w[u], x[u].z, acc.z);
        acc.w = fmaf(w[u], x[u].w, acc.w);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  const float inv = 1.f / wsum;
  if (col_ok) {
    uint2 packed;
    packed.x = ptx::pack_x2<F16>(acc.x * inv, acc.y * inv);
    packed.y = ptx::pack_x2<F16>(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(O + row * D + c4) = packed;
  }
  if (lane == 0) LSE[row] = m + logf(wsum);
}

template <int D, int MASK, bool F16>
static fa_status launch_tc_impl(const FwdArgs& a, int S, float* part_o, float* part_lse) {
  using C = TcCfg<D>;
  using Tile = TcTile<D>;
  auto kern = fa_fwd_tc_kernel<D, MASK, F16>;
  static bool attr_done[64] = {};  // per instantiation and device; benign race
  bool* done = device_flag(attr_done);
  if (done == nullptr || !*done) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return cuda_status(e);
    // the register split must fit the launch allocation, else setmaxnreg.inc
    // would wait forever: refuse to launch instead
    cudaFuncAttributes fattr;
    e = cudaFuncGetAttributes(&fattr, kern);
    if (e != cudaSuccess) return cuda_status(e);
    if (C::REGS_SPLIT > C::THREADS * fattr.numRegs) return FA_ERR_UNSUPPORTED;
    if (done != nullptr) *done = true;
  }
  CUtensorMap mq, mk, mv;
  CUresult r;
  if ((r = make_tmap_16bit(&mq, a.q, D, a.T, static_cast<long long>(a.B) * a.Hq, Tile::BOX_X,
                           Tile::TMA_SWIZZLE, F16)) != CUDA_SUCCESS)
    return cu_status(r);
  if ((r = make_tmap_16bit(&mk, a.k, D, a.T, static_cast<long long>(a.B) * a.Hkv, Tile::BOX_X,
                           Tile::TMA_SWIZZLE, F16)) != CUDA_SUCCESS)
    return cu_status(r);
  if ((r = make_tmap_16bit(&mv, a.v, D, a.T, static_cast<long long>(a.B) * a.Hkv, Tile::BOX_X,
                           Tile::TMA_SWIZZLE, F16)) != CUDA_SUCCESS)
    return cu_status(r);
  // packed global keys (local-global): the same boxes over [B*Hkv][rows][d];
  // otherwise K and V stand in (never read)
  CUtensorMap mkg = mk, mvg = mv;
  if (a.lg_packed) {
    if ((r = make_tmap_16bit(&mkg, a.lg_kg, D, a.lg_rows, static_cast<long long>(a.B) * a.Hkv,
                             Tile::BOX_X, Tile::TMA_SWIZZLE, F16)) != CUDA_SUCCESS)
      return cu_status(r);
    if ((r = make_tmap_16bit(&mvg, a.lg_vg, D, a.lg_rows, static_cast<long long>(a.B) * a.Hkv,
                             Tile::BOX_X, Tile::TMA_SWIZZLE, F16)) != CUDA_SUCCESS)
      return cu_status(r);
  }
  const long long units = static_cast<long long>(a.B) * a.Hq * ((a.T + 255) / 256) * S;
  const long long grid = units < tc_sm_count() ? units : tc_sm_count();  // one CTA per SM
  // scale * log2(e); never exactly 0, so that masked (infinite) scores give
  // exponents of -inf rather than NaN: for scale = 0 the smallest normal
  // float stands in, and every finite score's exponent still rounds to 0
  float scale_log2 = a.scale * 1.4426950408889634f;
  if (scale_log2 == 0.f) scale_log2 = 1.17549435e-38f;
  int wl, wr;
  effective_window(a, wl, wr);
  kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, a.stream>>>(
      mq, mk, mv, static_cast<uint16_t*>(a.o), a.lse, a.B, a.Hq, a.Hkv, a.T, scale_log2,
      static_cast<int>(units), S, S > 1 ? part_o : nullptr, S > 1 ? part_lse : nullptr, wl, wr,
      a.lg_bits, a.lg_list, a.lg_count, a.causal, mkg, mvg, a.lg_packed ? 1 : 0, a.lg_tokens,
      a.lg_ntok);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || S == 1) return cuda_status(e);
  // the merge, as a programmatic dependent launch: its grid may be scheduled
  // while the attention kernel finishes (every attention CTA signals that
  // at its start) and waits inside for that kernel's writes
  const long long rows = static_cast<long long>(a.B) * a.Hq * a.T;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows * 32 + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, fa_split_combine_kernel<F16>, static_cast<const float*>(part_o),
                         static_cast<const float*>(part_lse), static_cast<uint16_t*>(a.o), a.lse,
                         a.B * a.Hq, a.T, a.d, S, wl, wr);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(cudaGetLastError());
}

template <int MASK, bool F16>
static fa_status launch_tc_d(const FwdArgs& a, int S, float* po, float* pl) {
  switch (a.d) {
    case 16: return launch_tc_impl<16, MASK, F16>(a, S, po, pl);
    case 32: return launch_tc_impl<32, MASK, F16>(a, S, po, pl);
    case 64: return launch_tc_impl<64, MASK, F16>(a, S, po, pl);
    case 128: return launch_tc_impl<128, MASK, F16>(a, S, po, pl);
    default: return FA_ERR_UNSUPPORTED;
  }
}

template <bool F16>
static fa_status launch_tc_t(const FwdArgs& a, int S, float* po, float* pl) {
  int wl, wr;
  effective_window(a, wl, wr);
  if (a.local_global) return launch_tc_d<kMaskLocalGlobal, F16>(a, S, po, pl);
  if (wl < 0 && wr < 0) return launch_tc_d<kMaskNone, F16>(a, S, po, pl);
  if (wl < 0 && wr == 0) return launch_tc_d<kMaskCausal, F16>(a, S, po, pl);
  return launch_tc_d<kMaskBand, F16>(a, S, po, pl);
}

fa_status launch_tc(const FwdArgs& a) { return launch_tc_split(a, 1, nullptr, 0); }

fa_status launch_tc_split(const FwdArgs& a, int S, void* workspace, size_t workspace_bytes) {
  float* po = nullptr;
  float* pl = nullptr;
  if (S > 1) {
    const size_t need = split_workspace_bytes(a.B, a.Hq, a.T, a.d, S);
    if (workspace == nullptr || workspace_bytes < need) return FA_ERR_WORKSPACE;
    po = static_cast<float*>(workspace);
    pl = po + static_cast<size_t>(S) * a.B * a.Hq * a.T * a.d;
  }
  if (a.dtype == FA_DTYPE_BF16) return launch_tc_t<false>(a, S, po, pl);
  if (a.dtype == FA_DTYPE_F16) return launch_tc_t<true>(a, S, po, pl);
  return FA_ERR_UNSUPPORTED;
}

size_t split_workspace_bytes(int B, int Hq, int T, int d, int S) {
  // partial O (fp32) then partial LSE (fp32) of every split
  return static_cast<size_t>(S) * B * Hq * T * (static_cast<size_t>(d) + 1) * sizeof(float);
}

int split_heuristic(int B, int Hq, int T, int causal) {
  // split the KV range only when the row blocks leave more than half of the
  // SMs idle; then aim at about one unit per SM, with at least 4 KV tiles per
  // split (shorter ones are launch-latency bound and lose to the extra merge)
  const long long units = static_cast<long long>(B) * Hq * ((T + 255) / 256);
  const int sm = tc_sm_count();
  if (units * 2 > sm) return 1;
  const int n_all = (T + 127) / 128;
  long long s = (sm + units - 1) / units;
  if (s > n_all / 4) s = n_all / 4;
  if (s > kMaxSplits) s = kMaxSplits;
  (void)causal;
  return s < 2 ? 1 : static_cast<int>(s);
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
