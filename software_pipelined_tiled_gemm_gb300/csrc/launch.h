// launch.h -- host-side launchers, one per compiled kernel instance.  Each
// kernel lives in its own translation unit so the library builds in parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernel_params.h"

namespace spgemm {

#define SPGEMM_DECLARE_BN(BN)                                                              \
  cudaError_t gemm_set_smem_bn##BN(size_t smem);                                           \
  cudaError_t gemm_launch_bn##BN(const CUtensorMap& a, const CUtensorMap& b,               \
                                 const CUtensorMap& bt, const CUtensorMap& c,              \
                                 const CUtensorMap& bp, const Params& p, int grid,         \
                                 size_t smem, cudaStream_t stream);
SPGEMM_DECLARE_BN(64)
SPGEMM_DECLARE_BN(128)
SPGEMM_DECLARE_BN(256)
#undef SPGEMM_DECLARE_BN

// CTA-pair instances (cluster of 2, cta_group::2 MMAs, 256 x BN tiles).
#define SPGEMM_DECLARE_PAIR(BN)                                                            \
  cudaError_t gemm_set_smem_pair##BN(size_t smem);                                         \
  cudaError_t gemm_max_clusters_pair##BN(size_t smem, int* clusters);                      \
  cudaError_t gemm_launch_pair##BN(const CUtensorMap& a, const CUtensorMap& b,             \
                                   const CUtensorMap& bt, const CUtensorMap& c,            \
                                   const CUtensorMap& bp, const Params& p, int grid,       \
                                   size_t smem, cudaStream_t stream);
SPGEMM_DECLARE_PAIR(128)
SPGEMM_DECLARE_PAIR(256)
#undef SPGEMM_DECLARE_PAIR

// Copy the rows of A (M x K) and/or B (N x K) into zero-padded scratch with
// row pitch Kp (a multiple of 8 elements, so every row is 16-byte aligned).
cudaError_t launch_pad_operands(const uint16_t* A, int64_t M, uint16_t* Ap, const uint16_t* B,
                                int64_t N, uint16_t* Bp, int64_t K, int64_t Kp, int sm_count,
                                cudaStream_t stream);

// K = 0 with a bias: C[i, j] = epi(bias[j]) for an M x N C with pitch N
// (fp32, or the input type); bias holds N fp16/bf16 values.
cudaError_t launch_bias_fill(void* C, int64_t M, int64_t N, const void* bias, bool bf16,
                             int epilogue, bool out_f32, int sm_count, cudaStream_t stream);

}  // namespace spgemm
