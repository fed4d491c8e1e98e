// Epilogue stores of TMEM rows to row-major [token, head, d] 16-bit tensors.
//
// A tcgen05.ld 32x32b load leaves one TMEM lane -- one output row -- per thread,
// and rows of one head lie hq*d elements apart in memory. Were each thread to
// store its own 16 values as two 16-byte stores, every store instruction would
// touch 32 half-filled 32-byte sectors. Here adjacent lanes (rows r and r+1)
// swap half of their data first, so that the even lane stores the first 8 values
// and the odd lane the last 8 of the same row in the same instruction: each
// store instruction writes 16 whole sectors.
#pragma once

#include <stdint.h>

#include "sm103_ptx.cuh"

namespace teattn {

// Row pointer of this lane and of its pair partner (lane ^ 1); `valid` flags
// rows that may be written. Computed once per item.
template <typename T>
struct RowPair {
  T* lo;  // row of the even lane of the pair
  T* hi;  // row of the odd lane
  bool lo_ok, hi_ok;
};

template <typename T>
__device__ __forceinline__ RowPair<T> make_row_pair(T* own, bool own_ok) {
  const bool odd = threadIdx.x & 1;
  const unsigned long long mine = reinterpret_cast<unsigned long long>(own);
  const unsigned long long other = __shfl_xor_sync(0xffffffffu, mine, 1);
  const bool other_ok = __shfl_xor_sync(0xffffffffu, own_ok ? 1 : 0, 1) != 0;
  RowPair<T> r;
  r.lo = reinterpret_cast<T*>(odd ? other : mine);
  r.hi = reinterpret_cast<T*>(odd ? mine : other);
  r.lo_ok = odd ? other_ok : own_ok;
  r.hi_ok = odd ? own_ok : other_ok;
  return r;
}

// Store this lane's 16 fp32 values v (times scale) as 16-bit to columns
// [c0, c0+16) of its row; the pair partner takes part in the same call. Columns
// at or beyond d are not written. Every lane of the warp must call this.
template <bool kBF16, typename T>
__device__ __forceinline__ void store_pair16(const RowPair<T>& rp, int c0, int d, const uint32_t (&v)[16],
                                             float scale) {
  const bool odd = threadIdx.x & 1;
  uint4 first, second;
  first.x = pack2<kBF16>(__uint_as_float(v[0]) * scale, __uint_as_float(v[1]) * scale);
  first.y = pack2<kBF16>(__uint_as_float(v[2]) * scale, __uint_as_float(v[3]) * scale);
  first.z = pack2<kBF16>(__uint_as_float(v[4]) * scale, __uint_as_float(v[5]) * scale);
  first.w = pack2<kBF16>(__uint_as_float(v[6]) * scale, __uint_as_float(v[7]) * scale);
  second.x = pack2<kBF16>(__uint_as_float(v[8]) * scale, __uint_as_float(v[9]) * scale);
  second.y = pack2<kBF16>(__uint_as_float(v[10]) * scale, __uint_as_float(v[11]) * scale);
  second.z = pack2<kBF16>(__uint_as_float(v[12]) * scale, __uint_as_float(v[13]) * scale);
  second.w = pack2<kBF16>(__uint_as_float(v[14]) * scale, __uint_as_float(v[15]) * scale);
  // even lane hands over its last 8 values, odd lane its first 8
  const uint4 send = odd ? first : second;
  uint4 recv;
  recv.x = __shfl_xor_sync(0xffffffffu, send.x, 1);
  recv.y = __shfl_xor_sync(0xffffffffu, send.y, 1);
  recv.z = __shfl_xor_sync(0xffffffffu, send.z, 1);
  recv.w = __shfl_xor_sync(0xffffffffu, send.w, 1);
  const int col = c0 + (odd ? 8 : 0);
  if (col + 8 <= d) {
    // row of the even lane: first half from the even lane, second from the odd lane
    if (rp.lo_ok) *reinterpret_cast<uint4*>(rp.lo + col) = odd ? recv : first;
    // row of the odd lane
    if (rp.hi_ok) *reinterpret_cast<uint4*>(rp.hi + col) = odd ? second : recv;
  }
}

}  // namespace teattn
