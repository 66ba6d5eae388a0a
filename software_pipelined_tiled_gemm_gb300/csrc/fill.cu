// fill.cu -- C for an empty reduction (K = 0) with a bias:
//   C[i, j] = epi(bias[j]), rounded to C's type (or kept in fp32).
// Memory-bound; a grid-stride loop over C's elements.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "epilogue_math.cuh"
#include "launch.h"

namespace spgemm {

__global__ void __launch_bounds__(256) bias_fill_kernel(void* __restrict__ C, int64_t M, int64_t N,
                                                        const uint16_t* __restrict__ bias, int bf16,
                                                        int epilogue, int out_f32) {
  const int64_t total = M * N;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint16_t bits = bias[e % N];
    float v = bf16 ? __bfloat162float(__ushort_as_bfloat16(bits))
                   : __half2float(__ushort_as_half(bits));
    if (epilogue == 1) v = gelu_tanh(v);
    if (epilogue == 2) v = relu(v);
    if (out_f32)
      static_cast<float*>(C)[e] = v;
    else if (bf16)
      static_cast<__nv_bfloat16*>(C)[e] = __float2bfloat16_rn(v);
    else
      static_cast<__half*>(C)[e] = __float2half_rn(v);
  }
}

cudaError_t launch_bias_fill(void* C, int64_t M, int64_t N, const void* bias, bool bf16,
                             int epilogue, bool out_f32, int sm_count, cudaStream_t stream) {
  const int64_t total = M * N;
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  if (blocks > cap) blocks = cap;
  bias_fill_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(
      C, M, N, static_cast<const uint16_t*>(bias), bf16 ? 1 : 0, epilogue, out_f32 ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace spgemm
