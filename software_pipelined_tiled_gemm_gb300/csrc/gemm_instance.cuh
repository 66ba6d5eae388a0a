// gemm_instance.cuh -- defines the launcher pair of one kernel instance.
#pragma once

#include "gemm_kernel.cuh"
#include "launch.h"

#define SPGEMM_DEFINE_BN(BN)                                                                   \
  namespace spgemm {                                                                           \
  cudaError_t gemm_set_smem_bn##BN(size_t smem) {                                              \
    return cudaFuncSetAttribute(gemm_tn_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                static_cast<int>(smem));                                       \
  }                                                                                            \
  cudaError_t gemm_launch_bn##BN(const CUtensorMap& a, const CUtensorMap& b,                   \
                                 const CUtensorMap& c, const Params& p, int grid, size_t smem, \
                                 cudaStream_t stream) {                                        \
    gemm_tn_kernel<BN><<<grid, kThreads, smem, stream>>>(a, b, c, p);                          \
    return cudaGetLastError();                                                                 \
  }                                                                                            \
  }
