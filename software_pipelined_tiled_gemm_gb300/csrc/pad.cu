// pad.cu -- staging copy for operands whose rows cannot be described to the
// TMA engine (row pitch or base address not 16-byte aligned).
//
// dst[r, c] = src[r, c] for c < K and 0 for K <= c < Kp, Kp a multiple of 8.
// Memory-bound.  Each thread emits one 16-byte store of 8 elements.  Its 8
// source elements start at an arbitrary even byte address; they are taken
// from the two 16-byte-aligned words that cover them (two vector loads,
// shared with the neighbouring threads through L1) and shifted into place.
// Where an aligned word would reach outside the source array (its first or
// last few elements), the elements are read one by one instead.  Both
// operands are handled by one launch.
#include <cuda_runtime.h>

#include <cstdint>

#include "byte_shift.cuh"
#include "launch.h"

namespace spgemm {

__global__ void __launch_bounds__(256) pad_operands_kernel(const uint16_t* __restrict__ A, int64_t M,
                                                           uint16_t* __restrict__ Ap,
                                                           const uint16_t* __restrict__ B, int64_t N,
                                                           uint16_t* __restrict__ Bp, int64_t K,
                                                           int64_t Kp) {
  const int64_t vpr = Kp / 8;  // 16-byte vectors per padded row
  const int64_t nA = Ap ? M * vpr : 0;
  const int64_t nB = Bp ? N * vpr : 0;
  const int64_t total = nA + nB;
  for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < total;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const bool isA = v < nA;
    const int64_t w = isA ? v : v - nA;
    const int64_t r = w / vpr;
    const int64_t c0 = (w - r * vpr) * 8;
    const uint16_t* src = isA ? A : B;
    const int64_t rows = isA ? M : N;
    uint16_t* d = (isA ? Ap : Bp) + r * Kp + c0;
    const int64_t valid = K - c0 < 8 ? (K - c0 > 0 ? K - c0 : 0) : 8;  // in-row elements
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (valid > 0) {
      const uint16_t* s = src + r * K + c0;
      const uintptr_t addr = reinterpret_cast<uintptr_t>(s);
      const uintptr_t base = addr & ~static_cast<uintptr_t>(15);
      const uintptr_t first = reinterpret_cast<uintptr_t>(src);
      const uintptr_t end = reinterpret_cast<uintptr_t>(src + rows * K);  // one past the last element
      if (base >= first && base + 32 <= end) {  // both aligned words inside the array
        const uint4 lo = __ldg(reinterpret_cast<const uint4*>(base));
        const uint4 hi = __ldg(reinterpret_cast<const uint4*>(base + 16));
        out = shift_window(lo, hi, static_cast<uint32_t>(addr - base));
      } else {
        uint32_t wd[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < valid) wd[j >> 1] |= static_cast<uint32_t>(__ldg(s + j)) << ((j & 1) * 16);
        out = make_uint4(wd[0], wd[1], wd[2], wd[3]);
      }
      if (valid < 8) {  // zero the elements past the end of the row
        uint32_t wd[4] = {out.x, out.y, out.z, out.w};
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j >= valid) wd[j >> 1] &= (j & 1) ? 0x0000FFFFu : 0xFFFF0000u;
        out = make_uint4(wd[0], wd[1], wd[2], wd[3]);
      }
    }
    *reinterpret_cast<uint4*>(d) = out;
  }
}

cudaError_t launch_pad_operands(const uint16_t* A, int64_t M, uint16_t* Ap, const uint16_t* B,
                                int64_t N, uint16_t* Bp, int64_t K, int64_t Kp, int sm_count,
                                cudaStream_t stream) {
  const int64_t total = ((Ap ? M : 0) + (Bp ? N : 0)) * (Kp / 8);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(sm_count) * 16;
  if (blocks > cap) blocks = cap;
  pad_operands_kernel<<<static_cast<int>(blocks), threads, 0, stream>>>(A, M, Ap, B, N, Bp, K, Kp);
  return cudaGetLastError();
}

}  // namespace spgemm
