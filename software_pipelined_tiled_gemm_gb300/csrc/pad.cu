// pad.cu -- staging copy for operands whose rows cannot be described to the
// TMA engine (row pitch or base address not 16-byte aligned).
//
// dst[r, c] = src[r, c] for c < K and 0 for K <= c < Kp, Kp a multiple of 8.
// Memory-bound.  Each thread emits one 16-byte store of 8 elements per row,
// for kPadRows rows at a time.
// Its 8 source elements start at an arbitrary even byte address; they are
// taken from the two 16-byte-aligned words that cover them (two vector
// loads, shared with the neighbouring threads through L1) and shifted into
// place.
// Where an aligned word would reach outside the source array (its first or
// last few elements), the elements are read one by one instead.  Both
// operands are handled by one launch.
#include <cuda_runtime.h>

#include <cstdint>

#include "byte_shift.cuh"
#include "launch.h"

namespace spgemm {

constexpr int kPadThreads = 256;

// Rows a thread copies per step, their loads all issued before the first
// store, so that each thread keeps kPadRows x 2 loads in flight.
constexpr int kPadRows = 4;

// Zero the elements of `out` at and past `valid` (the end of the row).
__device__ __forceinline__ uint4 zero_past(uint4 out, int64_t valid) {
  uint32_t wd[4] = {out.x, out.y, out.z, out.w};
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j >= valid) wd[j >> 1] &= (j & 1) ? 0x0000FFFFu : 0xFFFF0000u;
  return make_uint4(wd[0], wd[1], wd[2], wd[3]);
}

// Grid: x over the 16-byte vectors of a padded row (kPadThreads per block),
// y over groups of kPadRows rows of A then B (striding by gridDim.y groups
// when there are more than a grid dimension holds), so a thread finds its
// rows and column without a division.
__global__ void __launch_bounds__(kPadThreads) pad_operands_kernel(
    const uint16_t* __restrict__ A, int64_t M, uint16_t* __restrict__ Ap,
    const uint16_t* __restrict__ B, int64_t N, uint16_t* __restrict__ Bp, int64_t K, int64_t Kp) {
  const int64_t v = static_cast<int64_t>(blockIdx.x) * kPadThreads + threadIdx.x;
  if (v >= Kp / 8) return;
  const int64_t rows_a = Ap ? M : 0;
  const int64_t rows = rows_a + (Bp ? N : 0);
  const int64_t c0 = v * 8;
  const int64_t valid = K - c0 < 8 ? (K - c0 > 0 ? K - c0 : 0) : 8;  // in-row elements
  for (int64_t row0 = static_cast<int64_t>(blockIdx.y) * kPadRows; row0 < rows;
       row0 += static_cast<int64_t>(gridDim.y) * kPadRows) {
    // Loads of every row of the group first: the two aligned words around
    // the row's 8 elements, when both lie inside the array.
    uint4 lo[kPadRows], hi[kPadRows];
    uint32_t shift[kPadRows];
    bool fast[kPadRows];
#pragma unroll
    for (int i = 0; i < kPadRows; ++i) {
      const int64_t row = row0 + i;
      fast[i] = false;
      shift[i] = 0u;
      lo[i] = hi[i] = make_uint4(0u, 0u, 0u, 0u);
      if (row < rows && valid > 0) {
        const bool isA = row < rows_a;
        const int64_t r = isA ? row : row - rows_a;
        const uint16_t* src = isA ? A : B;
        const int64_t nrows = isA ? M : N;
        const uintptr_t addr = reinterpret_cast<uintptr_t>(src + r * K + c0);
        const uintptr_t base = addr & ~static_cast<uintptr_t>(15);
        const uintptr_t first = reinterpret_cast<uintptr_t>(src);
        const uintptr_t end = reinterpret_cast<uintptr_t>(src + nrows * K);  // one past the last element
        if (base >= first && base + 32 <= end) {
          lo[i] = __ldg(reinterpret_cast<const uint4*>(base));
          hi[i] = __ldg(reinterpret_cast<const uint4*>(base + 16));
          shift[i] = static_cast<uint32_t>(addr - base);
          fast[i] = true;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kPadRows; ++i) {
      const int64_t row = row0 + i;
      if (row >= rows) break;
      const bool isA = row < rows_a;
      const int64_t r = isA ? row : row - rows_a;
      uint4 out = make_uint4(0u, 0u, 0u, 0u);
      if (valid > 0) {
        if (fast[i]) {
          out = shift_window(lo[i], hi[i], shift[i]);
        } else {  // an aligned word would reach outside the array: element by element
          const uint16_t* sp = (isA ? A : B) + r * K + c0;
          uint32_t wd[4] = {0u, 0u, 0u, 0u};
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (j < valid) wd[j >> 1] |= static_cast<uint32_t>(__ldg(sp + j)) << ((j & 1) * 16);
          out = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        }
        if (valid < 8) out = zero_past(out, valid);
      }
      *reinterpret_cast<uint4*>((isA ? Ap : Bp) + r * Kp + c0) = out;
    }
  }
}

cudaError_t launch_pad_operands(const uint16_t* A, int64_t M, uint16_t* Ap, const uint16_t* B,
                                int64_t N, uint16_t* Bp, int64_t K, int64_t Kp, int sm_count,
                                cudaStream_t stream) {
  (void)sm_count;
  const int64_t rows = (Ap ? M : 0) + (Bp ? N : 0);
  const int64_t vpr = Kp / 8;  // 16-byte vectors per padded row
  if (rows == 0 || vpr == 0) return cudaSuccess;
  const int64_t bx = (vpr + kPadThreads - 1) / kPadThreads;
  if (bx > 0x7fffffff) return cudaErrorInvalidValue;
  const int64_t groups = (rows + kPadRows - 1) / kPadRows;
  const dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(groups < 65535 ? groups : 65535));
  pad_operands_kernel<<<grid, kPadThreads, 0, stream>>>(A, M, Ap, B, N, Bp, K, Kp);
  return cudaGetLastError();
}

}  // namespace spgemm
