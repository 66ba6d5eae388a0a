// pad.cu -- staging copy for operands whose rows cannot be described to the
// TMA engine (row pitch or base address not 16-byte aligned).
//
// dst[r, c] = src[r, c] for c < K and 0 for K <= c < Kp, Kp a multiple of 8.
// Memory-bound: each thread emits one 16-byte store of 8 elements; source
// elements are read with 2-byte loads because source rows may start at any
// even address.  Both operands are handled by one launch.
#include <cuda_runtime.h>

#include <cstdint>

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
    const uint16_t* s = (isA ? A : B) + r * K;
    uint16_t* d = (isA ? Ap : Bp) + r * Kp + c0;
    uint32_t word[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t c = c0 + 2 * j;
      const uint32_t lo = c < K ? __ldg(s + c) : 0u;
      const uint32_t hi = c + 1 < K ? __ldg(s + c + 1) : 0u;
      word[j] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(d) = make_uint4(word[0], word[1], word[2], word[3]);
  }
}

cudaError_t launch_pad_operands(const uint16_t* A, int64_t M, uint16_t* Ap, const uint16_t* B,
                                int64_t N, uint16_t* Bp, int64_t K, int64_t Kp, int sm_count,
                                cudaStream_t stream) {
  const int64_t total = ((Ap ? M : 0) + (Bp ? N : 0)) * (Kp / 8);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  if (blocks > cap) blocks = cap;
  pad_operands_kernel<<<static_cast<int>(blocks), threads, 0, stream>>>(A, M, Ap, B, N, Bp, K, Kp);
  return cudaGetLastError();
}

}  // namespace spgemm
