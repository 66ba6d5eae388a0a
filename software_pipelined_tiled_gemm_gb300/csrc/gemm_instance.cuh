// gemm_instance.cuh -- defines the launchers of one kernel shape.  Each shape
// has four instances -- with or without the narrow-tile / stream-K code
// (kSplit), for B stored N x K or K x N (kKN) -- and more: for single-CTA
// shapes, with B's copies marked evict-first (kStream) and one or two K
// slices per ring slot (kSub); for CTA pairs, with two K slices per slot;
// and each with four or eight epilogue warps (kEpiG).  The launcher picks the
// one the plan's parameters need, so no instance carries a runtime branch on
// these choices in its copy, MMA and epilogue loops.
#pragma once

#include "gemm_kernel.cuh"
#include "launch.h"

namespace spgemm {

template <int BN, int CG, bool kStream, int kSub, int kEpiG>
cudaError_t set_smem_layouts(size_t smem) {
  const int bytes = static_cast<int>(smem);
  const cudaFuncAttribute attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e =
      cudaFuncSetAttribute(gemm_tn_kernel<BN, CG, false, false, kStream, kSub, kEpiG>, attr, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_tn_kernel<BN, CG, true, false, kStream, kSub, kEpiG>, attr, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_tn_kernel<BN, CG, false, true, kStream, kSub, kEpiG>, attr, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_tn_kernel<BN, CG, true, true, kStream, kSub, kEpiG>, attr, bytes);
  return e;
}

template <int BN, int CG, int kEpiG>
cudaError_t set_smem_groups(size_t smem) {
  cudaError_t e = set_smem_layouts<BN, CG, false, 1, kEpiG>(smem);
  if constexpr (CG == 1) {
    if (e == cudaSuccess) e = set_smem_layouts<BN, CG, true, 1, kEpiG>(smem);
    if (e == cudaSuccess) e = set_smem_layouts<BN, CG, true, 2, kEpiG>(smem);
  } else {
    if (e == cudaSuccess) e = set_smem_layouts<BN, CG, false, 2, kEpiG>(smem);
  }
  return e;
}

template <int BN, int CG>
cudaError_t set_smem_all(size_t smem) {
  cudaError_t e = set_smem_groups<BN, CG, 1>(smem);
  if (e == cudaSuccess) e = set_smem_groups<BN, CG, 2>(smem);
  return e;
}

template <int BN, int CG, bool kStream, int kSub, int kEpiG>
cudaError_t launch_layout(const cudaLaunchConfig_t& cfg, const CUtensorMap& a,
                          const CUtensorMap& b, const CUtensorMap& bt, const CUtensorMap& c,
                          const CUtensorMap& bp, const Params& p) {
  const bool split = p.tail_splits > 1 || p.sk_tiles > 0;
  if (p.b_kn) {
    if (split)
      return cudaLaunchKernelEx(&cfg, gemm_tn_kernel<BN, CG, true, true, kStream, kSub, kEpiG>, a,
                                b, bt, c, bp, p);
    return cudaLaunchKernelEx(&cfg, gemm_tn_kernel<BN, CG, false, true, kStream, kSub, kEpiG>, a, b,
                              bt, c, bp, p);
  }
  if (split)
    return cudaLaunchKernelEx(&cfg, gemm_tn_kernel<BN, CG, true, false, kStream, kSub, kEpiG>, a, b,
                              bt, c, bp, p);
  return cudaLaunchKernelEx(&cfg, gemm_tn_kernel<BN, CG, false, false, kStream, kSub, kEpiG>, a, b,
                            bt, c, bp, p);
}

// Picks the instance for the plan: narrow / stream-K code or not, B layout,
// evict-first B copies (single CTAs only), two K slices per ring slot (CTA
// pairs, and single CTAs streaming B), and the epilogue warps.
template <int BN, int CG, int kEpiG>
cudaError_t launch_groups(const cudaLaunchConfig_t& cfg, const CUtensorMap& a,
                          const CUtensorMap& b, const CUtensorMap& bt, const CUtensorMap& c,
                          const CUtensorMap& bp, const Params& p) {
  if constexpr (CG == 1) {
    if (p.b_stream && p.k_sub == 2)
      return launch_layout<BN, CG, true, 2, kEpiG>(cfg, a, b, bt, c, bp, p);
    if (p.b_stream) return launch_layout<BN, CG, true, 1, kEpiG>(cfg, a, b, bt, c, bp, p);
  } else {
    if (p.k_sub == 2) return launch_layout<BN, CG, false, 2, kEpiG>(cfg, a, b, bt, c, bp, p);
  }
  return launch_layout<BN, CG, false, 1, kEpiG>(cfg, a, b, bt, c, bp, p);
}

template <int BN, int CG>
cudaError_t launch_instance(const cudaLaunchConfig_t& cfg, const CUtensorMap& a,
                            const CUtensorMap& b, const CUtensorMap& bt, const CUtensorMap& c,
                            const CUtensorMap& bp, const Params& p) {
  if (p.epi_groups == 2) return launch_groups<BN, CG, 2>(cfg, a, b, bt, c, bp, p);
  return launch_groups<BN, CG, 1>(cfg, a, b, bt, c, bp, p);
}

// Launch configuration: `grid` CTAs of kernel_threads(epi_groups) threads,
// programmatic dependent launch allowed, and clusters of `cluster` (1 or 2)
// CTAs: 2 for pairs and for single CTAs whose tiles are split in two K halves
// within a cluster (Params::sk_cluster).
inline void make_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int cluster, int grid,
                        size_t smem, cudaStream_t stream, int epi_groups) {
  cfg = cudaLaunchConfig_t{};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kernel_threads(epi_groups == 2 ? 2 : 1), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  int n = 0;
  if (cluster == 2) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 2;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  cfg.attrs = attr;
  cfg.numAttrs = n;
}

}  // namespace spgemm

#define SPGEMM_DEFINE_BN(BN)                                                                   \
  namespace spgemm {                                                                           \
  cudaError_t gemm_set_smem_bn##BN(size_t smem) { return set_smem_all<BN, 1>(smem); }          \
  cudaError_t gemm_launch_bn##BN(const CUtensorMap& a, const CUtensorMap& b,                   \
                                 const CUtensorMap& bt, const CUtensorMap& c,                  \
                                 const CUtensorMap& bp, const Params& p, int grid, size_t smem, \
                                 cudaStream_t stream) {                                        \
    cudaLaunchConfig_t cfg;                                                                    \
    cudaLaunchAttribute attr[2];                                                               \
    make_config(cfg, attr, p.sk_cluster ? 2 : 1, grid, smem, stream, p.epi_groups);            \
    return launch_instance<BN, 1>(cfg, a, b, bt, c, bp, p);                                    \
  }                                                                                            \
  }

#define SPGEMM_DEFINE_PAIR(BN)                                                                 \
  namespace spgemm {                                                                           \
  cudaError_t gemm_set_smem_pair##BN(size_t smem) { return set_smem_all<BN, 2>(smem); }        \
  cudaError_t gemm_max_clusters_pair##BN(size_t smem, int* clusters) {                         \
    cudaLaunchConfig_t cfg;                                                                    \
    cudaLaunchAttribute attr[2];                                                               \
    make_config(cfg, attr, 2, 2, smem, nullptr, 1);                                            \
    return cudaOccupancyMaxActiveClusters(                                                     \
        clusters, gemm_tn_kernel<BN, 2, false, false, false, 1, 1>, &cfg);                     \
  }                                                                                            \
  cudaError_t gemm_launch_pair##BN(const CUtensorMap& a, const CUtensorMap& b,                 \
                                   const CUtensorMap& bt, const CUtensorMap& c,                \
                                   const CUtensorMap& bp, const Params& p, int grid,           \
                                   size_t smem, cudaStream_t stream) {                         \
    cudaLaunchConfig_t cfg;                                                                    \
    cudaLaunchAttribute attr[2];                                                               \
    make_config(cfg, attr, 2, grid, smem, stream, p.epi_groups);                               \
    return launch_instance<BN, 2>(cfg, a, b, bt, c, bp, p);                                    \
  }                                                                                            \
  }
