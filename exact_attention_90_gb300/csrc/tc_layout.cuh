// tc_layout.cuh -- tile geometry of the bf16 tensor-core attention kernel.
//
// One Q, K or V tile is ROWS (128, or 64 for the backward's query steps)
// rows x d columns of bf16, brought into shared memory by TMA as NBOX boxes
// of ROWS rows x BOX_X columns, back to back.  The
// box row is BOX_X * 2 bytes (32, 64 or 128) and uses the swizzle of the same
// width, so every 8-row group of a box is one swizzle atom of 8 * ROW_BYTES
// bytes.  The same bytes serve
//   * Q and K as K-major operands of S = Q K^T (the reduction runs over d,
//     which is contiguous): one MMA k-step covers 16 columns = 32 bytes of a
//     box row, so k-step kk sits in box kk / KSTEPS_PER_BOX at byte offset
//     (kk % KSTEPS_PER_BOX) * 32, and 8-row groups are SBO = 8 * ROW_BYTES
//     apart;
//   * V as the MN-major B operand of O += P V (the reduction runs over the
//     keys, which are the rows; d is contiguous): one k-step covers 16 rows =
//     16 * ROW_BYTES bytes of every box, 8-row groups are SBO apart and the
//     boxes (64-column atoms along d) are LBO = BOX_BYTES apart.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace fa {

template <int D, int ROWS_ = 128>
struct TcTile {
  static_assert(D == 16 || D == 32 || D == 64 || D == 128, "unsupported head dim");
  static_assert(ROWS_ == 128 || ROWS_ == 64, "tiles are 128 or 64 rows");
  static constexpr int ROWS = ROWS_;
  static constexpr int BOX_X = D < 64 ? D : 64;
  static constexpr int ROW_BYTES = BOX_X * 2;
  static constexpr int NBOX = D / BOX_X;
  static constexpr int BOX_BYTES = ROWS * ROW_BYTES;
  static constexpr int TILE_BYTES = NBOX * BOX_BYTES;
  static constexpr int KSTEPS_PER_BOX = ROW_BYTES / 32;
  static constexpr int QK_KSTEPS = D / 16;         // MMA k-steps of S = Q K^T
  static constexpr int PV_KSTEPS = ROWS / 16;      // MMA k-steps of O += P V
  static constexpr uint32_t SBO = 8 * ROW_BYTES;
  static constexpr uint32_t LAYOUT =
      ROW_BYTES == 128 ? ptx::kLayoutSw128 : (ROW_BYTES == 64 ? ptx::kLayoutSw64 : ptx::kLayoutSw32);
  // matching CUtensorMapSwizzle value: 1 = 32B, 2 = 64B, 3 = 128B
  static constexpr int TMA_SWIZZLE = ROW_BYTES == 128 ? 3 : (ROW_BYTES == 64 ? 2 : 1);

  // Descriptor halves.  A shared-memory address is below 2^18, so its 14-bit
  // start-address field never carries into the LBO field: the low word of a
  // k-step's descriptor is the tile's low word plus (byte offset >> 4).
  static constexpr uint32_t DESC_HI = (SBO >> 4) | (1u << 14) | (LAYOUT << 29);
  static constexpr uint32_t KM_LO_LBO = (16u >> 4) << 16;
  static constexpr uint32_t MN_LO_LBO = (static_cast<uint32_t>(BOX_BYTES) >> 4) << 16;
  __device__ static __forceinline__ uint32_t kmajor_lo(uint32_t base) {
    return (base >> 4) | KM_LO_LBO;
  }
  __device__ static __forceinline__ uint32_t mnmajor_lo(uint32_t base) {
    return (base >> 4) | MN_LO_LBO;
  }
  static constexpr uint32_t kmajor_step(int kk) {
    return static_cast<uint32_t>((kk / KSTEPS_PER_BOX) * BOX_BYTES + (kk % KSTEPS_PER_BOX) * 32) >> 4;
  }
  static constexpr uint32_t mnmajor_step(int kk) {
    return static_cast<uint32_t>(kk * 16 * ROW_BYTES) >> 4;
  }

  // K-major operand (Q or K tile at shared address `base`), k-step kk.
  __device__ static __forceinline__ uint64_t kmajor_desc(uint32_t base, int kk) {
    const uint32_t addr =
        base + (kk / KSTEPS_PER_BOX) * BOX_BYTES + (kk % KSTEPS_PER_BOX) * 32;
    return ptx::smem_desc(addr, 16, SBO, LAYOUT);
  }

  // MN-major operand (V tile at shared address `base`), k-step kk (16 rows).
  static constexpr uint32_t MN_LBO = BOX_BYTES;  // between 64-column atoms along d
  static constexpr uint32_t MN_SBO = SBO;        // between 8-row groups along the keys
  __device__ static __forceinline__ uint64_t mnmajor_desc(uint32_t base, int kk,
                                                          uint32_t lbo = MN_LBO,
                                                          uint32_t sbo = MN_SBO) {
    const uint32_t addr = base + kk * 16 * ROW_BYTES;
    return ptx::smem_desc(addr, lbo, sbo, LAYOUT);
  }
};

}  // namespace fa
