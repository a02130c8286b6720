// row_store.cuh -- epilogue stores of 16-bit rows, one row per lane.
//
// The tcgen05 kernels end with each thread holding one output row (its TMEM
// lane), lanes 2i and 2i+1 holding consecutive rows.  A 16-byte store per
// lane then touches 32 rows per warp instruction and half of each 32-byte
// sector.  Here the two lanes of a pair swap one 16-byte piece, so that each
// instruction writes whole sectors of two rows: the even lane the first half,
// the odd lane the second half, row r first, then row r + 1.
#pragma once

#include <cstdint>

namespace fa {

// The two rows of this lane's pair: the even row's pointer and which of the
// two exist (rows >= T are not written).
struct RowPair {
  uint16_t* even;  // row r of the pair (r = this lane's row minus lane & 1)
  uint16_t* odd;   // row r + 1
  bool ok_even, ok_odd;
  int odd_lane;    // lane & 1
};

// `base` is row 0 of the (batch, head) matrix, `ld` elements per row, `row`
// this lane's row.
__device__ __forceinline__ RowPair row_pair(uint16_t* base, int ld, int row, int T, int lane) {
  RowPair p;
  p.odd_lane = lane & 1;
  const int r = row - p.odd_lane;
  p.ok_even = r < T;
  p.ok_odd = r + 1 < T;
  p.even = base + static_cast<size_t>(p.ok_even ? r : 0) * ld;
  p.odd = p.ok_odd ? p.even + ld : p.even;
  return p;
}

// Store columns [col0, col0 + 16) of both rows of the pair (one 32-byte
// sector each): w[0..7] are this lane's row's 16 values as packed pairs.
// Every lane of the warp must call.
__device__ __forceinline__ void store_sector_pair(const RowPair& p, int col0, const uint32_t* w) {
  uint32_t rcv[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    rcv[e] = __shfl_xor_sync(0xffffffffu, p.odd_lane ? w[e] : w[4 + e], 1);
  const int piece = col0 + p.odd_lane * 8;
  if (p.ok_even)
    *reinterpret_cast<uint4*>(p.even + piece) =
        p.odd_lane ? make_uint4(rcv[0], rcv[1], rcv[2], rcv[3])
                   : make_uint4(w[0], w[1], w[2], w[3]);
  if (p.ok_odd)
    *reinterpret_cast<uint4*>(p.odd + piece) =
        p.odd_lane ? make_uint4(w[4], w[5], w[6], w[7])
                   : make_uint4(rcv[0], rcv[1], rcv[2], rcv[3]);
}

}  // namespace fa
