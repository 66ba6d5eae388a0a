// noalloc.cu -- gemm_run_noalloc: the GEMM for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or anything that allocates): code that
// runs under an allocator it does not own, a runtime that forbids
// allocations after start-up, or a path that must not add allocations while
// other work is being captured or scheduled.  gemm_run allocates twice: the
// plan's status word at plan creation, and scratch for padded copies of A and
// B when a row pitch or base address is not 16-byte aligned.  This entry
// point needs neither allocation.  Its scratch (the padded operands plus the
// kernel's status word) is one file-scope __device__ array of a fixed size,
// reserved by the CUDA module on every device that loads this library and
// held until the process exits.
//
// Host code must not use the array's name as a device address: on the host it
// names a host-side shadow, and a kernel given that address would fault (or,
// where the GPU can reach host memory, silently use the wrong memory).  The
// device address is taken with cudaGetSymbolAddress once per device, with
// that device current, during the set-up that the first call on each device
// performs.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/gemm.h"
#include "kernel_params.h"
#include "launch.h"
#include "ptx.cuh"

using namespace spgemm;

namespace {

constexpr size_t kStatusBytes = 256;  // status word area at the front of the scratch
constexpr size_t kScratchBytes = static_cast<size_t>(GEMM_NOALLOC_SCRATCH_BYTES);
constexpr int kMaxDevices = 64;

}  // namespace

// The scratch: [0, 256) status words, [256, ...) padded A then padded B.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kStatusBytes + kScratchBytes];

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceSetup {
  std::mutex mu;
  bool done = false;           // set only by a set-up that succeeded
  cudaError_t err = cudaSuccess;
  gemm_status_t status = GEMM_OK;
  uint8_t* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int sm_count = 0;
  int smem_optin = 0;
  EncodeTiledFn encode = nullptr;
};

DeviceSetup g_setup[kMaxDevices];

void setup_device(DeviceSetup& s, int dev) {
  // Runs with `dev` current, until it succeeds once on that device.
  s.status = GEMM_OK;
  s.err = cudaSuccess;
  cudaDeviceProp prop;
  s.err = cudaGetDeviceProperties(&prop, dev);
  if (s.err != cudaSuccess) { s.status = GEMM_ERR_CUDA; return; }
  if (prop.major != 10 || prop.minor != 3) { s.status = GEMM_ERR_UNSUPPORTED; return; }
  s.sm_count = prop.multiProcessorCount;
  s.err = cudaDeviceGetAttribute(&s.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (s.err != cudaSuccess) { s.status = GEMM_ERR_CUDA; return; }
  void* p = nullptr;
  s.err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (s.err != cudaSuccess || p == nullptr) { s.status = GEMM_ERR_CUDA; return; }
  s.scratch = static_cast<uint8_t*>(p);
  // Allow every kernel instance the largest dynamic shared memory it may use.
  const size_t lim = static_cast<size_t>(s.smem_optin);
  if ((s.err = gemm_set_smem_bn64(lim)) != cudaSuccess ||
      (s.err = gemm_set_smem_bn128(lim)) != cudaSuccess ||
      (s.err = gemm_set_smem_bn256(lim)) != cudaSuccess) {
    s.status = GEMM_ERR_CUDA;
    return;
  }
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  s.err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (s.err != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
    s.status = GEMM_ERR_CUDA;
    return;
  }
  s.encode = reinterpret_cast<EncodeTiledFn>(fn);
}

bool encode(const DeviceSetup& s, CUtensorMap* map, gemm_dtype_t dt, const void* base,
            int64_t inner, int64_t rows, int64_t pitch, uint32_t box_inner, uint32_t box_rows,
            CUtensorMapL2promotion l2) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch) * 2u};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return s.encode(map,
                  dt == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, l2,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (!na || !nb) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

extern "C" gemm_status_t gemm_run_noalloc(const void* A, const void* B, void* C, int64_t M,
                                          int64_t N, int64_t K, gemm_dtype_t dtype,
                                          gemm_epilogue_t epi, int stages, void* stream_handle) {
  constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return GEMM_ERR_INVALID_ARG;
  if ((dtype != GEMM_F16 && dtype != GEMM_BF16) ||
      (epi != GEMM_EPI_NONE && epi != GEMM_EPI_GELU_TANH && epi != GEMM_EPI_RELU) || stages < 1 ||
      stages > kMaxStages)
    return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_OK;
  if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;
  const size_t bytesA = static_cast<size_t>(M) * K * 2, bytesB = static_cast<size_t>(N) * K * 2;
  const size_t bytesC = static_cast<size_t>(M) * N * 2;
  if (overlap(C, bytesC, A, bytesA) || overlap(C, bytesC, B, bytesB)) return GEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
       reinterpret_cast<uintptr_t>(C)) & 1u)
    return GEMM_ERR_INVALID_ARG;

  const bool padA = (K % 8) != 0 || (reinterpret_cast<uintptr_t>(A) & 15u) != 0;
  const bool padB = (K % 8) != 0 || (reinterpret_cast<uintptr_t>(B) & 15u) != 0;
  const int64_t Kp = (K + 7) / 8 * 8;
  const size_t need = ((padA ? M : 0) + (padB ? N : 0)) * static_cast<size_t>(Kp) * 2;
  if (K > 0 && need > kScratchBytes) return GEMM_ERR_INVALID_ARG;  // beyond the static scratch

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED;
  DeviceSetup& s = g_setup[dev];
  {
    // A failed set-up is not kept: the next call on this device tries again
    // (the failure may have been transient, e.g. an error left over from
    // earlier work, or a first call made during a stream capture).
    std::lock_guard<std::mutex> lock(s.mu);
    if (!s.done) {
      setup_device(s, dev);
      if (s.status != GEMM_OK) return s.status;
      s.done = true;
    }
  }

  cudaStream_t stream = static_cast<cudaStream_t>(stream_handle);
  if (K == 0) return cudaMemsetAsync(C, 0, bytesC, stream) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;

  // Tile width: the widest whose ring fits, narrowed while it leaves SMs idle.
  const int cands[3] = {256, 128, 64};
  int bn = 0, bufs = 0;
  size_t smem = 0;
  const int64_t tm = (M + kBM - 1) / kBM;
  for (int i = 0; i < 3; ++i) {
    int b = 2;
    size_t need_smem = kernel_smem_bytes(cands[i], stages, b);
    if (need_smem > static_cast<size_t>(s.smem_optin)) {
      b = 1;
      need_smem = kernel_smem_bytes(cands[i], stages, b);
    }
    if (need_smem > static_cast<size_t>(s.smem_optin)) continue;
    bn = cands[i];
    bufs = b;
    smem = need_smem;
    if (tm * ((N + bn - 1) / bn) >= s.sm_count) break;
  }
  if (bn == 0) return GEMM_ERR_SMEM_BUDGET;

  int* status = reinterpret_cast<int*>(s.scratch);
  uint16_t* Ap = padA ? reinterpret_cast<uint16_t*>(s.scratch + kStatusBytes) : nullptr;
  uint16_t* Bp = padB ? reinterpret_cast<uint16_t*>(s.scratch + kStatusBytes) + (padA ? M * Kp : 0)
                      : nullptr;
  // The status word must start at zero; the padded copies are fully rewritten.
  if (cudaMemsetAsync(status, 0, kStatusBytes, stream) != cudaSuccess) return GEMM_ERR_CUDA;
  if (padA || padB) {
    if (launch_pad_operands(static_cast<const uint16_t*>(A), M, Ap,
                            static_cast<const uint16_t*>(B), N, Bp, K, Kp, s.sm_count,
                            stream) != cudaSuccess)
      return GEMM_ERR_CUDA;
  }
  const void* effA = padA ? static_cast<const void*>(Ap) : A;
  const void* effB = padB ? static_cast<const void*>(Bp) : B;
  const int64_t Keff = (padA || padB) ? Kp : K;
  const bool tma_store = (N % 8) == 0 && (reinterpret_cast<uintptr_t>(C) & 15u) == 0;

  CUtensorMap tmA, tmB, tmC;
  std::memset(&tmC, 0, sizeof(tmC));
  if (!encode(s, &tmA, dtype, effA, Keff, M, Keff, kBK, kBM, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
      !encode(s, &tmB, dtype, effB, Keff, N, Keff, kBK, static_cast<uint32_t>(bn),
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
      (tma_store && !encode(s, &tmC, dtype, C, N, M, N, kStoreCols, 32, CU_TENSOR_MAP_L2_PROMOTION_NONE)))
    return GEMM_ERR_CUDA;

  Params p;
  std::memset(&p, 0, sizeof(p));
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(Keff);
  p.tiles_m = static_cast<int>(tm);
  p.tiles_n = static_cast<int>((N + bn - 1) / bn);
  const int64_t tiles = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
  if (tiles > kMaxDim) return GEMM_ERR_INVALID_ARG;
  p.num_tiles = static_cast<int>(tiles);
  p.k_blocks = static_cast<int>((Keff + kBK - 1) / kBK);
  p.stages = stages;
  p.num_acc = 2;
  p.tmem_cols = std::max(32, bn * 2);
  p.raster_group = static_cast<int>(std::min<int64_t>(16, tm));
  p.store_bufs = bufs;
  p.epi_groups = 1;
  p.bf16 = dtype == GEMM_BF16 ? 1 : 0;
  p.epilogue = static_cast<int>(epi);
  p.out_f32 = 0;
  p.tma_store = tma_store ? 1 : 0;
  p.idesc = ptx::instr_desc_f16(kBM, bn, dtype == GEMM_BF16);
  p.C = C;
  p.ldc = N;
  p.status = status;
  p.timeout_ns = 2000000000ull;
  p.dp_tiles = p.num_tiles;  // every tile whole
  p.tail_splits = 1;
  p.num_units = p.num_tiles;
  p.idesc_tail = p.idesc;
  p.a_box_rows = kBM;
  const int grid = static_cast<int>(std::min<int64_t>(tiles, s.sm_count));
  cudaError_t e;
  switch (bn) {
    case 64: e = gemm_launch_bn64(tmA, tmB, tmB, tmC, tmB, p, grid, smem, stream); break;
    case 128: e = gemm_launch_bn128(tmA, tmB, tmB, tmC, tmB, p, grid, smem, stream); break;
    default: e = gemm_launch_bn256(tmA, tmB, tmB, tmC, tmB, p, grid, smem, stream); break;
  }
  return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}
