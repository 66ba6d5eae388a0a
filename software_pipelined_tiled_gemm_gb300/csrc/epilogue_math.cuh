// epilogue_math.cuh -- the epilogue functions' arithmetic on an fp32 value,
// shared by the GEMM epilogue and the K = 0 bias fill so both evaluate the
// same formula.
#pragma once

namespace spgemm {

// tanh-GELU as the Triton lecture notes ("GeLU") and the XLA:GPU emitters
// page (loop-emitter example, @gelu) write it:
//   0.5 x (1 + tanh(u)), u = 0.7978845608 (x + 0.044715 x^3),
// evaluated as the identical x / (1 + exp(-2u)), which cannot produce
// inf/inf for large |u| (x -> x for u -> +inf, x -> -0 for u -> -inf).
// CUDA's fast exponential and division keep the epilogue cheap; their
// few-ulp fp32 error is far below the 8/11-bit precision of the rounded
// output, and __fdividef(x, inf) gives -0/+0.
__device__ __forceinline__ float gelu_tanh(float x) {
  const float inner = x * fmaf(0.044715f, x * x, 1.0f);
  return __fdividef(x, 1.0f + __expf(-1.5957691216f * inner));
}

// ReLU: max(x, 0), with -0 and NaN giving +0.
__device__ __forceinline__ float relu(float x) { return x > 0.0f ? x : 0.0f; }

}  // namespace spgemm
