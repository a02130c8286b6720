// fa_unit.cu -- single-tile test kernels for the PTX building blocks of the
// bf16 attention kernel (contracts in include/fa_unit.h).  Each uses exactly
// the tile geometry, descriptors and instruction encodings of fa_tc.cu, one
// block at a time, so a wrong bit field shows up as a wrong number here.
#include "fa_internal.h"
#include "../../include/fa_unit.h"
#include "ptx.cuh"
#include "tc_layout.cuh"
#include "wait.cuh"

namespace fa {

static __device__ unsigned int g_unit_err;

namespace {

// zeroed bytes after the unit kernels' tiles (absorbs reads through a wrong
// descriptor stride)
constexpr int kUnitPad = 64 * 1024;

template <int D>
struct UnitSmem {
  static constexpr int BYTES = 1024 + TcTile<D>::TILE_BYTES + TcTile<128>::TILE_BYTES + kUnitPad + 128;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                    ~static_cast<uintptr_t>(1023));
}

template <int D>
__global__ void __launch_bounds__(128) unit_tma_kernel(const __grid_constant__ CUtensorMap tm,
                                                       uint4* out) {
  using Tile = TcTile<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 2 * Tile::TILE_BYTES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 1);
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    ptx::mbar_arrive_expect_tx(bar, Tile::TILE_BYTES);
    for (int bx = 0; bx < Tile::NBOX; ++bx)
      ptx::tma_load_3d(sm + bx * Tile::BOX_BYTES, &tm, bar, bx * 64, 0, 0);
  }
  const bool ok = wait_bar(bar, 0, abort_flag, &g_unit_err, kErrWaitLoad);
  if (!ok && threadIdx.x == 0) drain_bar(bar, 0, &g_unit_err);
  __syncthreads();
  const uint4* src = reinterpret_cast<const uint4*>(sm);
  for (int i = threadIdx.x; i < Tile::TILE_BYTES / 16; i += 128) out[i] = src[i];
}

template <int D>
__global__ void __launch_bounds__(128) unit_qk_kernel(const __grid_constant__ CUtensorMap tq,
                                                      const __grid_constant__ CUtensorMap tk,
                                                      float* s_out) {
  using Tile = TcTile<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sQ = sm;
  uint8_t* sK = sm + Tile::TILE_BYTES;
  uint64_t* bar_ld = reinterpret_cast<uint64_t*>(sm + 2 * Tile::TILE_BYTES);
  uint64_t* bar_mma = bar_ld + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_ld, 1);
    ptx::mbar_init(bar_mma, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(tmem_slot, 128);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) {
    ptx::mbar_arrive_expect_tx(bar_ld, 2 * Tile::TILE_BYTES);
    for (int bx = 0; bx < Tile::NBOX; ++bx) {
      ptx::tma_load_3d(sQ + bx * Tile::BOX_BYTES, &tq, bar_ld, bx * 64, 0, 0);
      ptx::tma_load_3d(sK + bx * Tile::BOX_BYTES, &tk, bar_ld, bx * 64, 0, 0);
    }
    if (wait_bar(bar_ld, 0, abort_flag, &g_unit_err, kErrWaitMma)) {
      ptx::tc_fence_after();
      constexpr uint32_t IDESC = ptx::idesc_bf16(128, 128, false, false);
      for (int kk = 0; kk < Tile::QK_KSTEPS; ++kk)
        ptx::mma_ss(tmem, Tile::kmajor_desc(ptx::smem_u32(sQ), kk),
                    Tile::kmajor_desc(ptx::smem_u32(sK), kk), IDESC, kk > 0 ? 1u : 0u);
      ptx::mma_commit(bar_mma);
      drain_bar(bar_mma, 0, &g_unit_err);
    } else {
      drain_bar(bar_ld, 0, &g_unit_err);
    }
  }
  __syncwarp();
  const bool ok = __all_sync(0xffffffffu, wait_bar(bar_mma, 0, abort_flag, &g_unit_err,
                                                   kErrWaitSoftmax));
  ptx::tc_fence_after();
  if (ok) {
    const int row = warp * 32 + lane;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    for (int c = 0; c < 4; ++c) {
      uint32_t r[32];
      ptx::tmem_ld32(taddr + c * 32, r);
      ptx::tmem_ld_wait(r);
      for (int u = 0; u < 32; ++u) s_out[row * 128 + c * 32 + u] = __uint_as_float(r[u]);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 0) ptx::tmem_dealloc(tmem, 128);
}

template <int D>
__global__ void __launch_bounds__(128)
    unit_pv_kernel(const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tp,
                   const float* p_in, float* o_out, int mode, uint32_t lbo, uint32_t sbo) {
  using Tile = TcTile<D>;
  using PTile = TcTile<128>;  // P as a 128 x 128 K-major bf16 operand (mode 2)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sV = sm;
  uint8_t* sP = sm + Tile::TILE_BYTES;
  uint8_t* sEnd = sP + PTile::TILE_BYTES + kUnitPad;
  uint64_t* bar_ld = reinterpret_cast<uint64_t*>(sEnd);
  uint64_t* bar_mma = bar_ld + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = warp * 32 + lane;
  // zero the tiles and the padding after them: a descriptor that points
  // outside the loaded bytes then reads zeros, not stale data
  for (uint8_t* z = sm + threadIdx.x * 16; z < sEnd; z += 128 * 16)
    *reinterpret_cast<uint4*>(z) = make_uint4(0u, 0u, 0u, 0u);
  ptx::fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_ld, 1);
    ptx::mbar_init(bar_mma, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(tmem_slot, 256);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // P at columns [0, 64), O at [128, 128 + D)
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  if (threadIdx.x == 0) {
    ptx::mbar_arrive_expect_tx(bar_ld, Tile::TILE_BYTES + (mode == 2 ? PTile::TILE_BYTES : 0));
    for (int bx = 0; bx < Tile::NBOX; ++bx)
      ptx::tma_load_3d(sV + bx * Tile::BOX_BYTES, &tv, bar_ld, bx * 64, 0, 0);
    if (mode == 2)
      for (int bx = 0; bx < PTile::NBOX; ++bx)
        ptx::tma_load_3d(sP + bx * PTile::BOX_BYTES, &tp, bar_ld, bx * 64, 0, 0);
  }
  {
    // zero all 256 columns of this warp's lanes, then write P (two bf16 per
    // column) into columns [0, 64)
    uint32_t zero[32];
    for (int u = 0; u < 32; ++u) zero[u] = 0u;
    for (int c = 0; c < 8; ++c) ptx::tmem_st32(tmem + lane_off + c * 32, zero);
    ptx::tmem_st_wait();
    if (mode != 2) {
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
        for (int u = 0; u < 16; ++u)
          pk[u] = ptx::pack_bf16x2(p_in[row * 128 + c * 32 + 2 * u],
                                   p_in[row * 128 + c * 32 + 2 * u + 1]);
        ptx::tmem_st16(tmem + lane_off + c * 16, pk);
      }
      ptx::tmem_st_wait();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (mode == 3) {
    // round trip: read the packed P columns back
    for (int c = 0; c < 2; ++c) {
      uint32_t r[32];
      ptx::tmem_ld32(tmem + lane_off + c * 32, r);
      ptx::tmem_ld_wait(r);
      for (int u = 0; u < 32; ++u) o_out[row * 64 + c * 32 + u] = __uint_as_float(r[u]);
    }
    if (threadIdx.x == 0) drain_bar(bar_ld, 0, &g_unit_err);
  } else {
    if (threadIdx.x == 0) {
      if (wait_bar(bar_ld, 0, abort_flag, &g_unit_err, kErrWaitMma)) {
        ptx::tc_fence_after();
        constexpr uint32_t IDESC_PV = ptx::idesc_bf16(128, D, false, true);
        const uint32_t aV = ptx::smem_u32(sV);
        const uint32_t L = lbo ? lbo : Tile::MN_LBO;
        const uint32_t S = sbo ? sbo : Tile::MN_SBO;
        for (int kk = 0; kk < Tile::PV_KSTEPS; ++kk) {
          if (mode == 2)
            ptx::mma_ss(tmem + 128, PTile::kmajor_desc(ptx::smem_u32(sP), kk),
                        Tile::mnmajor_desc(aV, kk, L, S), IDESC_PV, kk > 0 ? 1u : 0u);
          else
            ptx::mma_ts(tmem + 128, tmem + kk * 8, Tile::mnmajor_desc(aV, kk, L, S), IDESC_PV,
                        kk > 0 ? 1u : 0u);
        }
        if (mode == 1) {
          // overwrite the P columns right away, as the attention kernel's next
          // S = Q K^T does; the P.V result above must be unaffected
          constexpr uint32_t IDESC_QK = ptx::idesc_bf16(128, 128, false, false);
          for (int kk = 0; kk < Tile::QK_KSTEPS; ++kk)
            ptx::mma_ss(tmem, Tile::kmajor_desc(aV, kk), Tile::kmajor_desc(aV, kk), IDESC_QK,
                        kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(bar_mma);
        drain_bar(bar_mma, 0, &g_unit_err);
      } else {
        drain_bar(bar_ld, 0, &g_unit_err);
      }
    }
    __syncwarp();
    const bool ok = __all_sync(0xffffffffu, wait_bar(bar_mma, 0, abort_flag, &g_unit_err,
                                                     kErrWaitSoftmax));
    ptx::tc_fence_after();
    if (ok) {
      for (int c = 0; c < D / 32 + (D < 32 ? 1 : 0); ++c) {
        uint32_t r[32];
        ptx::tmem_ld32(tmem + lane_off + 128 + c * 32, r);
        ptx::tmem_ld_wait(r);
        for (int u = 0; u < 32 && c * 32 + u < D; ++u)
          o_out[row * D + c * 32 + u] = __uint_as_float(r[u]);
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 0) ptx::tmem_dealloc(tmem, 256);
}

// A wait that can never complete: nothing arrives on the barrier.  Every
// thread must give up after `budget` clocks, record the timeout and exit.
__global__ void __launch_bounds__(128) unit_timeout_kernel(long long budget, int* gave_up) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const bool ok = wait_bar(&bar, 0, &abort_flag, &g_unit_err, kErrWaitSoftmax, budget);
  // once the flag is up, a later wait returns at once
  const bool ok2 = wait_bar(&bar, 0, &abort_flag, &g_unit_err, kErrWaitSoftmax, budget);
  if (!ok && !ok2) atomicAdd(gave_up, 1);
}

fa_status check_unit_ptrs(int d, std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs) {
    if (!p) return FA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(p) & 15u) return FA_ERR_MISALIGNED;
  }
  if (d != 16 && d != 32 && d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

template <int D>
fa_status set_smem(const void* kern) {
  return cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          UnitSmem<D>::BYTES));
}

template <int D>
fa_status unit_tma_impl(const void* x, void* out, cudaStream_t st) {
  using Tile = TcTile<D>;
  CUtensorMap m;
  CUresult r = make_tmap_bf16(&m, x, D, 128, 1, Tile::BOX_X, Tile::TMA_SWIZZLE);
  if (r != CUDA_SUCCESS) return cu_status(r);
  fa_status s = set_smem<D>(reinterpret_cast<const void*>(unit_tma_kernel<D>));
  if (s != FA_OK) return s;
  unit_tma_kernel<D><<<1, 128, UnitSmem<D>::BYTES, st>>>(m, static_cast<uint4*>(out));
  return cuda_status(cudaGetLastError());
}

template <int D>
fa_status unit_qk_impl(const void* q, const void* k, float* s, cudaStream_t st) {
  using Tile = TcTile<D>;
  CUtensorMap mq, mk;
  CUresult r = make_tmap_bf16(&mq, q, D, 128, 1, Tile::BOX_X, Tile::TMA_SWIZZLE);
  if (r == CUDA_SUCCESS) r = make_tmap_bf16(&mk, k, D, 128, 1, Tile::BOX_X, Tile::TMA_SWIZZLE);
  if (r != CUDA_SUCCESS) return cu_status(r);
  fa_status e = set_smem<D>(reinterpret_cast<const void*>(unit_qk_kernel<D>));
  if (e != FA_OK) return e;
  unit_qk_kernel<D><<<1, 128, UnitSmem<D>::BYTES, st>>>(mq, mk, s);
  return cuda_status(cudaGetLastError());
}

template <int D>
fa_status unit_pv_impl(const float* p, const void* pb, const void* v, float* o, int mode,
                       unsigned lbo, unsigned sbo, cudaStream_t st) {
  using Tile = TcTile<D>;
  CUtensorMap mv, mp;
  CUresult r = make_tmap_bf16(&mv, v, D, 128, 1, Tile::BOX_X, Tile::TMA_SWIZZLE);
  if (r == CUDA_SUCCESS)
    r = make_tmap_bf16(&mp, pb ? pb : v, pb ? 128 : D, 128, 1, pb ? 64 : Tile::BOX_X,
                       pb ? TcTile<128>::TMA_SWIZZLE : Tile::TMA_SWIZZLE);
  if (r != CUDA_SUCCESS) return cu_status(r);
  fa_status e = set_smem<D>(reinterpret_cast<const void*>(unit_pv_kernel<D>));
  if (e != FA_OK) return e;
  unit_pv_kernel<D><<<1, 128, UnitSmem<D>::BYTES, st>>>(mv, mp, p, o, mode, lbo, sbo);
  return cuda_status(cudaGetLastError());
}

// Pipe-rate probe: every thread runs 8 independent dependency chains of one
// instruction kind for `iters` rounds, so that the pipe, not the latency of
// one chain, sets the pace.  Kinds: 0 = ex2.approx.ftz.f32 on the
// special-function unit (x <- 2^-x, which stays in [0.5, 1]); 1 = scalar fp32
// FMA; 2 = paired fp32 FMA (fma.rn.f32x2, two FMAs per instruction).  Each
// CTA records its clock64 span; the dynamic shared memory the launch asks
// for keeps one CTA per SM.
constexpr int kRateThreads = 512;
constexpr int kRateChains = 8;
constexpr int kRateSmem = 160 * 1024;

template <int KIND>
__global__ void __launch_bounds__(kRateThreads) unit_pipe_rate_kernel(int iters, float* sink,
                                                                      long long* cycles) {
  float x[kRateChains];
#pragma unroll
  for (int i = 0; i < kRateChains; ++i) x[i] = 0.5f + 0.01f * (threadIdx.x & 7) + 0.003f * i;
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
    if constexpr (KIND == 0) {
#pragma unroll
      for (int i = 0; i < kRateChains; ++i) x[i] = ptx::ex2(-x[i]);
    } else if constexpr (KIND == 1) {
#pragma unroll
      for (int i = 0; i < kRateChains; ++i) x[i] = fmaf(x[i], 0.999f, 0.001f);
    } else {
      const uint64_t a2 = ptx::f2_pack(0.999f, 0.999f), b2 = ptx::f2_pack(0.001f, 0.001f);
#pragma unroll
      for (int i = 0; i < kRateChains; i += 2) {
        const uint64_t y = ptx::fma2(ptx::f2_pack(x[i], x[i + 1]), a2, b2);
        ptx::f2_unpack(y, x[i], x[i + 1]);
      }
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kRateChains; ++i) acc += x[i];
  if (acc == 12345.f) sink[threadIdx.x] = acc;  // keeps the chains live
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

template <int KIND>
fa_status unit_pipe_rate_launch(int iters, int blocks, float* sink, long long* cycles,
                                cudaStream_t st) {
  auto kern = unit_pipe_rate_kernel<KIND>;
  static bool attr_done[64] = {};
  bool* done = device_flag(attr_done);
  if (done == nullptr || !*done) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kRateSmem);
    if (e != cudaSuccess) return cuda_status(e);
    if (done != nullptr) *done = true;
  }
  kern<<<blocks, kRateThreads, kRateSmem, st>>>(iters, sink, cycles);
  return cuda_status(cudaGetLastError());
}

fa_status unit_timeout_impl(long long budget, int* gave_up, cudaStream_t st) {
  unit_timeout_kernel<<<1, 128, 0, st>>>(budget, gave_up);
  return cuda_status(cudaGetLastError());
}

}  // namespace

fa_status unit_read_and_clear_error(unsigned int* word) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_unit_err, sizeof(v));
  if (e != cudaSuccess) return cuda_status(e);
  if (v) {
    e = cudaMemcpyToSymbol(g_unit_err, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_status(e);
  }
  *word = v;
  return FA_OK;
}

}  // namespace fa

extern "C" {

fa_status fa_unit_tma(const void* x, void* out, int d, void* stream) {
  fa_status s = fa::check_unit_ptrs(d, {x, out});
  if (s != FA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (d) {
    case 16: return fa::unit_tma_impl<16>(x, out, st);
    case 32: return fa::unit_tma_impl<32>(x, out, st);
    case 64: return fa::unit_tma_impl<64>(x, out, st);
    default: return fa::unit_tma_impl<128>(x, out, st);
  }
}

fa_status fa_unit_qk(const void* q, const void* k, float* s_out, int d, void* stream) {
  fa_status s = fa::check_unit_ptrs(d, {q, k, s_out});
  if (s != FA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (d) {
    case 16: return fa::unit_qk_impl<16>(q, k, s_out, st);
    case 32: return fa::unit_qk_impl<32>(q, k, s_out, st);
    case 64: return fa::unit_qk_impl<64>(q, k, s_out, st);
    default: return fa::unit_qk_impl<128>(q, k, s_out, st);
  }
}

fa_status fa_unit_pv(const float* p, const void* pb, const void* v, float* o, int d, int mode,
                     unsigned lbo, unsigned sbo, void* stream) {
  fa_status s = fa::check_unit_ptrs(d, {v, o});
  if (s != FA_OK) return s;
  if (mode < 0 || mode > 3) return FA_ERR_INVALID_ARG;
  if (mode == 2 ? pb == nullptr : p == nullptr) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(pb)) & 15u)
    return FA_ERR_MISALIGNED;
  if ((lbo | sbo) & 15u || lbo >= (1u << 18) || sbo >= (1u << 18)) return FA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (d) {
    case 16: return fa::unit_pv_impl<16>(p, pb, v, o, mode, lbo, sbo, st);
    case 32: return fa::unit_pv_impl<32>(p, pb, v, o, mode, lbo, sbo, st);
    case 64: return fa::unit_pv_impl<64>(p, pb, v, o, mode, lbo, sbo, st);
    default: return fa::unit_pv_impl<128>(p, pb, v, o, mode, lbo, sbo, st);
  }
}

fa_status fa_unit_pipe_rate(int kind, int iters, int blocks, float* sink, long long* cycles,
                            void* stream) {
  if (!sink || !cycles || iters < 1 || iters > (1 << 24) || blocks < 1 || blocks > 4096)
    return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(sink) & 3u) || (reinterpret_cast<uintptr_t>(cycles) & 7u))
    return FA_ERR_MISALIGNED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (kind) {
    case 0: return fa::unit_pipe_rate_launch<0>(iters, blocks, sink, cycles, st);
    case 1: return fa::unit_pipe_rate_launch<1>(iters, blocks, sink, cycles, st);
    case 2: return fa::unit_pipe_rate_launch<2>(iters, blocks, sink, cycles, st);
    default: return FA_ERR_INVALID_ARG;
  }
}

fa_status fa_unit_timeout(long long budget_cycles, int* gave_up, void* stream) {
  if (!gave_up || budget_cycles < 1 || budget_cycles > (1ll << 31)) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(gave_up) & 3u) return FA_ERR_MISALIGNED;
  return fa::unit_timeout_impl(budget_cycles, gave_up, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
