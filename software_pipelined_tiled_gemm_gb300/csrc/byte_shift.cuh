// byte_shift.cuh -- a 16-byte window at an even byte offset of two adjacent
// 16-byte words; used by the staging copy (pad.cu) to realign source rows
// and by the GEMM epilogue to realign C rows whose pitch is not a multiple
// of 16 bytes.
#pragma once

#include <cstdint>

namespace spgemm {

// Bytes [off, off + 16) of the 32-byte little-endian value (lo, hi), off even.
__device__ __forceinline__ uint4 shift_window(const uint4& lo, const uint4& hi, uint32_t off) {
  const uint32_t q = off >> 2;          // whole 32-bit words to skip (0..3)
  const uint32_t sh = (off & 3u) * 8u;  // then 0 or 16 more bits
  uint32_t a0, a1, a2, a3, a4;
  switch (q) {
    case 0: a0 = lo.x; a1 = lo.y; a2 = lo.z; a3 = lo.w; a4 = hi.x; break;
    case 1: a0 = lo.y; a1 = lo.z; a2 = lo.w; a3 = hi.x; a4 = hi.y; break;
    case 2: a0 = lo.z; a1 = lo.w; a2 = hi.x; a3 = hi.y; a4 = hi.z; break;
    default: a0 = lo.w; a1 = hi.x; a2 = hi.y; a3 = hi.z; a4 = hi.w; break;
  }
  return make_uint4(__funnelshift_r(a0, a1, sh), __funnelshift_r(a1, a2, sh),
                    __funnelshift_r(a2, a3, sh), __funnelshift_r(a3, a4, sh));
}

}  // namespace spgemm
