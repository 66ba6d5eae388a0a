// gemm_instance.cuh -- defines the launchers of one kernel shape (both the
// plain instance and the one that can run narrow tail tiles).
#pragma once

#include "gemm_kernel.cuh"
#include "launch.h"

#define SPGEMM_DEFINE_BN(BN)                                                                   \
  namespace spgemm {                                                                           \
  cudaError_t gemm_set_smem_bn##BN(size_t smem) {                                              \
    cudaError_t e = cudaFuncSetAttribute(gemm_tn_kernel<BN, 1, false>,                         \
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,          \
                                         static_cast<int>(smem));                              \
    if (e != cudaSuccess) return e;                                                            \
    return cudaFuncSetAttribute(gemm_tn_kernel<BN, 1, true>,                                   \
                                cudaFuncAttributeMaxDynamicSharedMemorySize,                   \
                                static_cast<int>(smem));                                       \
  }                                                                                            \
  cudaError_t gemm_launch_bn##BN(const CUtensorMap& a, const CUtensorMap& b,                   \
                                 const CUtensorMap& bt, const CUtensorMap& c, const CUtensorMap& bp, \
                                 const Params& p, int grid, size_t smem, cudaStream_t stream) {                 \
    cudaLaunchConfig_t cfg = cudaLaunchConfig_t{};                                             \
    cudaLaunchAttribute attr[1];                                                               \
    cfg.gridDim = dim3(grid, 1, 1);                                                            \
    cfg.blockDim = dim3(kThreads, 1, 1);                                                       \
    cfg.dynamicSmemBytes = smem;                                                               \
    cfg.stream = stream;                                                                       \
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;                           \
    attr[0].val.programmaticStreamSerializationAllowed = 1;                                    \
    cfg.attrs = attr;                                                                          \
    cfg.numAttrs = 1;                                                                          \
    if (p.tail_splits > 1 || p.sk_tiles > 0)                                                   \
      return cudaLaunchKernelEx(&cfg, gemm_tn_kernel<BN, 1, true>, a, b, bt, c, bp, p);            \
    return cudaLaunchKernelEx(&cfg, gemm_tn_kernel<BN, 1, false>, a, b, bt, c, bp, p);             \
  }                                                                                            \
  }

#define SPGEMM_DEFINE_PAIR(BN)                                                                  \
  namespace spgemm {                                                                            \
  cudaError_t gemm_set_smem_pair##BN(size_t smem) {                                             \
    cudaError_t e = cudaFuncSetAttribute(gemm_tn_kernel<BN, 2, false>,                          \
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,           \
                                         static_cast<int>(smem));                               \
    if (e != cudaSuccess) return e;                                                             \
    return cudaFuncSetAttribute(gemm_tn_kernel<BN, 2, true>,                                    \
                                cudaFuncAttributeMaxDynamicSharedMemorySize,                    \
                                static_cast<int>(smem));                                        \
  }                                                                                             \
  static void pair_config_##BN(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int grid,    \
                               size_t smem, cudaStream_t stream) {                              \
    cfg = cudaLaunchConfig_t{};                                                                 \
    cfg.gridDim = dim3(grid, 1, 1);                                                             \
    cfg.blockDim = dim3(kThreads, 1, 1);                                                        \
    cfg.dynamicSmemBytes = smem;                                                                \
    cfg.stream = stream;                                                                        \
    attr[0].id = cudaLaunchAttributeClusterDimension;                                           \
    attr[0].val.clusterDim.x = 2;                                                               \
    attr[0].val.clusterDim.y = 1;                                                               \
    attr[0].val.clusterDim.z = 1;                                                               \
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;                            \
    attr[1].val.programmaticStreamSerializationAllowed = 1;                                     \
    cfg.attrs = attr;                                                                           \
    cfg.numAttrs = 2;                                                                           \
  }                                                                                             \
  cudaError_t gemm_max_clusters_pair##BN(size_t smem, int* clusters) {                          \
    cudaLaunchConfig_t cfg;                                                                     \
    cudaLaunchAttribute attr[2];                                                                \
    pair_config_##BN(cfg, attr, 2, smem, nullptr);                                              \
    return cudaOccupancyMaxActiveClusters(clusters, gemm_tn_kernel<BN, 2, false>, &cfg);        \
  }                                                                                             \
  cudaError_t gemm_launch_pair##BN(const CUtensorMap& a, const CUtensorMap& b,                  \
                                   const CUtensorMap& bt, const CUtensorMap& c, const CUtensorMap& bp, \
                                   const Params& p, int grid, size_t smem, cudaStream_t stream) {                          \
    cudaLaunchConfig_t cfg;                                                                     \
    cudaLaunchAttribute attr[2];                                                                \
    pair_config_##BN(cfg, attr, grid, smem, stream);                                            \
    if (p.tail_splits > 1 || p.sk_tiles > 0)                                                                      \
      return cudaLaunchKernelEx(&cfg, gemm_tn_kernel<BN, 2, true>, a, b, bt, c, bp, p);                 \
    return cudaLaunchKernelEx(&cfg, gemm_tn_kernel<BN, 2, false>, a, b, bt, c, bp, p);                  \
  }                                                                                             \
  }
