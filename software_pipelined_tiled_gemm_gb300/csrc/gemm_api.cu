// gemm_api.cu -- the C ABI declared in include/gemm.h: argument checking,
// tile/ring planning, tensor-map encoding, launches and error reporting.
//
// The planner follows the TileLang tutorial's shared-memory budget
// (pipelined_gemm.py, shared_bytes(): stages * (block_M*block_K +
// block_N*block_K) * element size, checked against the device limit the way
// its main() marks a depth "OVER"), plus the epilogue staging and barrier
// bytes this kernel adds on top.
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "../../include/gemm.h"
#include "kernel_params.h"
#include "launch.h"
#include "ptx.cuh"

using namespace spgemm;

namespace {

thread_local std::string g_last_error;

gemm_status_t fail(gemm_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

gemm_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(GEMM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Restores the caller's current device on scope exit.
struct DeviceGuard {
  int prev = -1;
  bool switched = false;
  cudaError_t err = cudaSuccess;
  explicit DeviceGuard(int dev) {
    err = cudaGetDevice(&prev);
    if (err == cudaSuccess && prev != dev) {
      err = cudaSetDevice(dev);
      switched = err == cudaSuccess;
    }
  }
  ~DeviceGuard() {
    if (switched) cudaSetDevice(prev);
  }
};

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s per wait

}  // namespace

// gemm_run_host splits problems of at least kHostPanelMinBytes of copies into
// blocks of C: up to kHostPanelsMax row panels and as many column panels, each
// at least kHostPanelMinRows rows / columns (smaller blocks run as GEMMs too
// short to keep the SMs busy: 4096^3 took 0.526 ms in 16 blocks of 1024,
// 0.487 ms in 4 of 2048).
constexpr int kHostPanelsMax = 4;
constexpr int64_t kHostPanelMinRows = 1536;
constexpr size_t kHostPanelMinBytes = 32u << 20;

// Automatic stream-K also needs the last, partial wave to leave each walker
// idle for at least this many K slices: (1 - leftover tiles / walkers) x K.
constexpr int kStreamKMinIdleSlices = 24;

struct gemm_plan {
  int device = 0;
  int64_t M = 0, N = 0, K = 0;
  gemm_dtype_t dtype = GEMM_F16;
  gemm_epilogue_t epi = GEMM_EPI_NONE;
  int stages = 0;                // as requested (runs must pass the same value)
  int ring_stages = 0;           // K slices in flight actually built (<= stages)
  gemm_variant_t variant = GEMM_PIPELINED;

  int sm_count = 0;
  int cg = 1;                    // CTAs per output tile (2 = CTA pair)
  int bn = 256;
  int num_acc = 2;
  int store_bufs = 2;
  int raster_group = 16;
  int grid = 0;
  int max_ctas = 0;
  int64_t tiles_m = 0, tiles_n = 0, num_tiles = 0;
  size_t smem = 0;
  unsigned long long timeout_ns = kDefaultTimeoutNs;
  int debug_fault = 0;
  int out_f32 = 0;               // C element: 0 = input type, 1 = fp32
  int b_kn = 0;                  // B stored K x N (read MN-major)
  int k_sub = 1;                 // 64-wide K slices per ring slot
  int epi_groups = 1;            // epilogue column groups (1: 4 warps, 2: 8 warps)
  int k_serpentine = 0;          // odd waves walk K downwards
  int l2_prefetch_first = 0;     // prefetch the first ring's slices before the PDL wait
  int sk_cluster = 0;            // K halves exchanged within 2-CTA clusters
  int sk_first = 0;              // stream-K share before the whole tiles
  // C's row pitch in elements when it differs from N: the block plans of
  // gemm_run_host write a block of a wider C (0 = N).
  int64_t ldc = 0;

  int* d_status = nullptr;       // [0] code, [1] detail
  int64_t dp_tiles = 0;          // tiles run whole
  int tail_splits = 1;           // narrow tiles per tail tile (cut along N)
  int64_t num_units = 0;
  int64_t sk_tiles = 0;          // stream-K tiles after dp_tiles
  float* sk_ws = nullptr;        // fp32 partials of stream-K tiles
  int* sk_flags = nullptr;       // partial-ready flags (reset by the owner)
  uint16_t* scratch = nullptr;   // padded copies of A and/or B
  size_t scratch_bytes = 0;

  // tensor-map cache, keyed by the pointers/pitches they were encoded for
  const void* mapA_ptr = nullptr;
  const void* mapB_ptr = nullptr;
  const void* mapC_ptr = nullptr;
  int64_t mapK = -1;
  CUtensorMap tmA{}, tmB{}, tmBt{}, tmC{};   // tmBt: B box of a narrow tail tile
  CUtensorMap tmBp{};                        // B, unswizzled 4-slice box, for L2 prefetch
  int prefetch_kb = 0;

  // device staging for gemm_run_host
  void* hA = nullptr;
  void* hB = nullptr;
  void* hC = nullptr;
  // gemm_run_host pipelining (see gemm_run_host): blocks of C, panel_rows x
  // panel_cols (shorter at the ends), each run by a block plan of its own
  // (blk[last row panel][last column panel]); copies in on one stream, in the
  // order the blocks can start, and out on a second.
  gemm_tuning_t tuning{};
  bool has_tuning = false;
  int64_t panel_rows = 0;          // 0: no blocks yet chosen
  int64_t panel_cols = 0;
  int num_panels = 0;              // row panels
  int num_col_panels = 0;          // column panels
  gemm_plan* blk[2][2] = {{nullptr, nullptr}, {nullptr, nullptr}};
  cudaStream_t copy_in = nullptr;
  cudaStream_t copy_out = nullptr;
  cudaEvent_t ev_start = nullptr, ev_done = nullptr;
  cudaEvent_t ev_a[kHostPanelsMax] = {}, ev_b[kHostPanelsMax] = {};
  cudaEvent_t ev_c[kHostPanelsMax * kHostPanelsMax] = {};

  int last_pads = 0;
  int last_tma_store = 0;
  int last_kernels = 0;
};

namespace {

gemm_status_t encode_2d(CUtensorMap* map, gemm_dtype_t dt, const void* base, int64_t inner,
                        int64_t rows, int64_t pitch_elems, uint32_t box_inner, uint32_t box_rows,
                        CUtensorMapL2promotion l2,
                        CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch_elems) * 2u};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estride[2] = {1, 1};
  const CUtensorMapDataType t =
      dt == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = enc(map, t, 2, const_cast<void*>(base), dims, strides, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d) for %lld x %lld",
                static_cast<int>(r), static_cast<long long>(rows), static_cast<long long>(inner));
  return GEMM_OK;
}

// K x N B (row pitch `cols` elements, `rows` rows; cols % 64 == 0 and
// rows % 8 == 0) viewed as (64 columns, 8 rows, cols / 64 column blocks,
// rows / 8 row groups), box (64, 8, blocks, 8): one box is a 64-row K slice
// of `blocks` 64-column blocks, written to shared memory as 1024-byte atoms
// in the order [row group][column block].
gemm_status_t encode_b_kn(CUtensorMap* map, gemm_dtype_t dt, const void* base, int64_t cols,
                          int64_t rows, uint32_t blocks) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  const cuuint64_t dims[4] = {64u, 8u, static_cast<cuuint64_t>(cols / 64),
                              static_cast<cuuint64_t>(rows / 8)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(cols) * 2u, 128u,
                                 static_cast<cuuint64_t>(cols) * 16u};
  const cuuint32_t box[4] = {64u, 8u, blocks, static_cast<cuuint32_t>(kBK / 8)};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  const CUtensorMapDataType t =
      dt == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = enc(map, t, 4, const_cast<void*>(base), dims, strides, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled (K x N B) failed (CUresult %d)",
                static_cast<int>(r));
  return GEMM_OK;
}

// fp32 C: 2-D map with 4-byte elements, 128-byte swizzle (box rows of 128 B).
gemm_status_t encode_2d_f32(CUtensorMap* map, const void* base, int64_t inner, int64_t rows,
                            int64_t pitch_elems, uint32_t box_inner, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch_elems) * 4u};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estride[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides,
                   box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled (fp32 C) failed (CUresult %d)",
                static_cast<int>(r));
  return GEMM_OK;
}

gemm_status_t check_common(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                           gemm_epilogue_t epi, int stages) {
  if (M < 0 || N < 0 || K < 0)
    return fail(GEMM_ERR_INVALID_ARG, "negative size M=%lld N=%lld K=%lld", (long long)M,
                (long long)N, (long long)K);
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return fail(GEMM_ERR_INVALID_ARG, "size above 2^31-1");
  if (dtype != GEMM_F16 && dtype != GEMM_BF16)
    return fail(GEMM_ERR_INVALID_ARG, "dtype %d out of range", static_cast<int>(dtype));
  if (epi != GEMM_EPI_NONE && epi != GEMM_EPI_GELU_TANH && epi != GEMM_EPI_RELU)
    return fail(GEMM_ERR_INVALID_ARG, "epilogue %d out of range", static_cast<int>(epi));
  if (stages < 1 || stages > kMaxStages)
    return fail(GEMM_ERR_INVALID_ARG, "stages %d outside [1, %d]", stages, kMaxStages);
  return GEMM_OK;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

cudaError_t set_smem(int bn, int cg, size_t smem) {
  if (cg == 2) return bn == 128 ? gemm_set_smem_pair128(smem) : gemm_set_smem_pair256(smem);
  switch (bn) {
    case 64: return gemm_set_smem_bn64(smem);
    case 128: return gemm_set_smem_bn128(smem);
    default: return gemm_set_smem_bn256(smem);
  }
}

cudaError_t launch(int bn, int cg, const CUtensorMap& a, const CUtensorMap& b,
                   const CUtensorMap& bt, const CUtensorMap& c, const CUtensorMap& bp,
                   const Params& p, int grid, size_t smem, cudaStream_t s) {
  if (cg == 2)
    return bn == 128 ? gemm_launch_pair128(a, b, bt, c, bp, p, grid, smem, s)
                     : gemm_launch_pair256(a, b, bt, c, bp, p, grid, smem, s);
  switch (bn) {
    case 64: return gemm_launch_bn64(a, b, bt, c, bp, p, grid, smem, s);
    case 128: return gemm_launch_bn128(a, b, bt, c, bp, p, grid, smem, s);
    default: return gemm_launch_bn256(a, b, bt, c, bp, p, grid, smem, s);
  }
}

}  // namespace

extern "C" {

const char* gemm_status_string(gemm_status_t s) {
  switch (s) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
    case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED";
    case GEMM_ERR_SMEM_BUDGET: return "GEMM_ERR_SMEM_BUDGET";
    case GEMM_ERR_PLAN_MISMATCH: return "GEMM_ERR_PLAN_MISMATCH";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
    case GEMM_ERR_BOUNDS: return "GEMM_ERR_BOUNDS";
  }
  return "GEMM_ERR_UNKNOWN";
}

static_assert(GEMM_WAIT_PRODUCER_EMPTY == kDetailProducerEmpty &&
                  GEMM_WAIT_PRODUCER_DRAIN == kDetailProducerDrain &&
                  GEMM_WAIT_MMA_ACC_EMPTY == kDetailMmaAccEmpty && GEMM_WAIT_MMA_FULL == kDetailMmaFull &&
                  GEMM_WAIT_MMA_DRAIN == kDetailMmaDrain && GEMM_WAIT_EPI_FULL == kDetailEpiFull &&
                  GEMM_WAIT_SK_FLAG == kDetailSkFlag && GEMM_WAIT_SK_COPY == kDetailSkCopy &&
                  GEMM_WAIT_SK_FREE == kDetailSkFree,
              "gemm_wait_t must match the kernel's wait identifiers");
static_assert(GEMM_ERR_BOUNDS == kStatusBounds && GEMM_ERR_TIMEOUT == kStatusTimeout &&
                  GEMM_CHECK_SMEM_LAYOUT == kCheckSmemLayout && GEMM_CHECK_TILE == kCheckTile &&
                  GEMM_CHECK_K_SLICE == kCheckKSlice && GEMM_CHECK_TMA_COORD == kCheckTmaCoord &&
                  GEMM_CHECK_MMA_TMEM == kCheckMmaTmem && GEMM_CHECK_MMA_SLOT == kCheckMmaSlot &&
                  GEMM_CHECK_EPI_TMEM == kCheckEpiTmem && GEMM_CHECK_STAGING == kCheckStaging &&
                  GEMM_CHECK_STORE == kCheckStore && GEMM_CHECK_PARTIAL == kCheckPartial &&
                  GEMM_CHECK_FIXUP == kCheckFixup,
              "gemm_check_t must match the kernel's check identifiers");

int gemm_bounds_checked(void) { return SPGEMM_BOUNDS_CHECKS ? 1 : 0; }

const char* gemm_wait_detail_string(int32_t detail) {
  switch (detail) {
    case 0: return "";
    case GEMM_WAIT_PRODUCER_EMPTY: return "TMA producer waiting for a free ring slot";
    case GEMM_WAIT_PRODUCER_DRAIN: return "TMA producer waiting for its last copies to land";
    case GEMM_WAIT_MMA_ACC_EMPTY: return "MMA issuer waiting for the epilogue to free an accumulator";
    case GEMM_WAIT_MMA_FULL: return "MMA issuer waiting for a ring slot's copies";
    case GEMM_WAIT_MMA_DRAIN: return "MMA issuer waiting for its last MMAs to complete";
    case GEMM_WAIT_EPI_FULL: return "epilogue waiting for an accumulator to be filled";
    case GEMM_WAIT_SK_FLAG: return "stream-K owner waiting for its partner's partial";
    case GEMM_WAIT_SK_COPY: return "stream-K owner waiting for the partial's bytes";
    case GEMM_WAIT_SK_FREE: return "cluster split contributor waiting for the owner's ring";
    case GEMM_CHECK_SMEM_LAYOUT: return "ring, staging and barriers exceed the launch's shared memory";
    case GEMM_CHECK_TILE: return "tile index or tile coordinates out of range";
    case GEMM_CHECK_K_SLICE: return "K slot outside the unit's range or the K extent";
    case GEMM_CHECK_TMA_COORD: return "copy coordinate out of range or unaligned";
    case GEMM_CHECK_MMA_TMEM: return "accumulator columns beyond the TMEM allocation";
    case GEMM_CHECK_MMA_SLOT: return "ring slot index beyond the ring";
    case GEMM_CHECK_EPI_TMEM: return "epilogue TMEM columns beyond the allocation";
    case GEMM_CHECK_STAGING: return "staging buffer beyond the warp's staging area";
    case GEMM_CHECK_STORE: return "C block outside the tile grid or unaligned";
    case GEMM_CHECK_PARTIAL: return "stream-K workspace slot beyond the workspace";
    case GEMM_CHECK_FIXUP: return "stream-K partial region beyond the ring";
  }
  return "unknown wait";
}

const char* gemm_last_error(void) { return g_last_error.c_str(); }

const char* gemm_version(void) { return "0.1.0"; }

size_t gemm_smem_bytes(int bm, int bn, int bk, int elem_bytes, int stages) {
  if (bm <= 0 || bn <= 0 || bk <= 0 || elem_bytes <= 0 || stages <= 0) return 0;
  return static_cast<size_t>(stages) *
         (static_cast<size_t>(bm) * bk + static_cast<size_t>(bn) * bk) *
         static_cast<size_t>(elem_bytes);
}

namespace {

// Tuning requests, validated (0 = choose).
struct Wants {
  int bn = 0, group = 0, ctas = 0, cg = 0, split = 0;
  unsigned long long timeout = kDefaultTimeoutNs;
};

// Checks everything about a plan request that needs no device.
gemm_status_t check_create_args(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                                gemm_epilogue_t epi, int stages, gemm_variant_t variant,
                                const gemm_tuning_t* tuning, Wants* w) {
  gemm_status_t st = check_common(M, N, K, dtype, epi, stages);
  if (st != GEMM_OK) return st;
  if (variant != GEMM_PIPELINED && variant != GEMM_SINGLE_BUFFER)
    return fail(GEMM_ERR_INVALID_ARG, "variant %d out of range", static_cast<int>(variant));
  if (variant == GEMM_SINGLE_BUFFER && stages != 1)
    return fail(GEMM_ERR_INVALID_ARG, "the single-buffer variant has exactly 1 stage (got %d)",
                stages);
  if (tuning) {
    w->bn = tuning->tile_n;
    w->group = tuning->raster_group;
    w->ctas = tuning->max_ctas;
    w->cg = tuning->cta_group;
    w->split = tuning->tail_split;
    if (w->split < -1 || w->split > kMaxTailSplits)
      return fail(GEMM_ERR_INVALID_ARG, "tail_split %d not in {-1, 0, 1, 2, 3, 4}", w->split);
    if (w->bn != 0 && w->bn != 64 && w->bn != 128 && w->bn != 256)
      return fail(GEMM_ERR_INVALID_ARG, "tile_n %d not in {0, 64, 128, 256}", w->bn);
    if (w->cg < 0 || w->cg > 2)
      return fail(GEMM_ERR_INVALID_ARG, "cta_group %d not in {0, 1, 2}", w->cg);
    if (w->cg == 2 && w->bn == 64)
      return fail(GEMM_ERR_INVALID_ARG, "CTA pairs use tile_n 128 or 256");
    if (w->group < 0 || w->ctas < 0)
      return fail(GEMM_ERR_INVALID_ARG, "negative raster_group / max_ctas");
    if (tuning->timeout_ns < 0) return fail(GEMM_ERR_INVALID_ARG, "negative timeout_ns");
    if (tuning->debug_fault < 0 || tuning->debug_fault > 2)
      return fail(GEMM_ERR_INVALID_ARG, "debug_fault %d not in {0, 1, 2}", tuning->debug_fault);
    if (tuning->debug_fault == 2 && !SPGEMM_BOUNDS_CHECKS)
      return fail(GEMM_ERR_INVALID_ARG,
                  "debug_fault 2 forces a range check to fail; only the bounds-checked build "
                  "has the checks");
    if (tuning->out_f32 < 0 || tuning->out_f32 > 1)
      return fail(GEMM_ERR_INVALID_ARG, "out_f32 %d not in {0, 1}", tuning->out_f32);
    if (tuning->b_kn < 0 || tuning->b_kn > 1)
      return fail(GEMM_ERR_INVALID_ARG, "b_kn %d not in {0, 1}", tuning->b_kn);
    if (tuning->epi_groups < 0 || tuning->epi_groups > 2)
      return fail(GEMM_ERR_INVALID_ARG, "epi_groups %d not in {0, 1, 2}", tuning->epi_groups);
    if (tuning->k_serpentine < -1 || tuning->k_serpentine > 1)
      return fail(GEMM_ERR_INVALID_ARG, "k_serpentine %d not in {-1, 0, 1}",
                  tuning->k_serpentine);
    if (tuning->b_kn == 1 && w->split >= 2)
      return fail(GEMM_ERR_INVALID_ARG, "narrow tail tiles are not available with b_kn = 1");
    if (tuning->timeout_ns > 0) w->timeout = static_cast<unsigned long long>(tuning->timeout_ns);
  }
  return GEMM_OK;
}

// Co-resident 2-CTA clusters of the pair kernel of tile width bn with `smem`
// bytes of dynamic shared memory per CTA.
using PairClustersFn = gemm_status_t (*)(void* ctx, int bn, size_t smem, int* clusters);

// From the device: ctx points to the device's opt-in shared-memory limit.
gemm_status_t cuda_pair_clusters(void* ctx, int bn, size_t smem, int* clusters) {
  cudaError_t e = set_smem(bn, 2, *static_cast<const size_t*>(ctx));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic smem)");
  e = bn == 128 ? gemm_max_clusters_pair128(smem, clusters)
                : gemm_max_clusters_pair256(smem, clusters);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveClusters");
  return GEMM_OK;
}

// From a description: ctx points to a gemm_device_desc_t.  Every kernel
// instance runs one CTA per SM (its registers allow no second one), so the
// count does not depend on the tile width or the shared memory.
gemm_status_t desc_pair_clusters(void* ctx, int, size_t, int* clusters) {
  *clusters = static_cast<const gemm_device_desc_t*>(ctx)->pair_clusters;
  return GEMM_OK;
}

// Properties of the current device (which must be `device`) that the
// planner uses, except pair_clusters.  GEMM_ERR_UNSUPPORTED unless sm_103.
gemm_status_t device_props(int device, gemm_device_desc_t* desc) {
  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
  if (prop.major != 10 || prop.minor != 3)
    return fail(GEMM_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                device, prop.major, prop.minor);
  int smem_optin = 0;
  e = cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(smem optin)");
  desc->sm_count = prop.multiProcessorCount;
  desc->smem_optin = smem_optin;
  desc->l2_bytes = prop.l2CacheSize;
  desc->pair_clusters = 0;
  return GEMM_OK;
}

// The planner: chooses the tile, ring, epilogue, walkers and last-wave
// treatment of a plan for a device described by `dev`, and fills the
// corresponding fields of *p.  Host arithmetic only, except what
// `pair_clusters` does; allocates nothing (on failure *p is left to the
// caller to discard).
// Rows of A one K slice of the ring holds: all kBM rows of the CTA's tile,
// or 64 for single-CTA tiles when M <= 64 (then a single row of tiles, run by
// the evict-first-B instances, which size their A slices from the box).
int ring_a_rows(int cta_group, int64_t M) { return (cta_group == 1 && M <= 64) ? 64 : kBM; }

gemm_status_t plan_layout(gemm_plan* p, const gemm_device_desc_t& dev,
                          PairClustersFn pair_clusters, void* ctx, int64_t M, int64_t N,
                          int64_t K, gemm_dtype_t dtype, gemm_epilogue_t epi, int stages,
                          gemm_variant_t variant, const gemm_tuning_t* tuning, const Wants& w) {
  const int want_bn = w.bn, want_group = w.group, want_ctas = w.ctas, want_cg = w.cg,
            want_split = w.split;
  // Tile shape.  Candidates in order of preference: CTA pairs (256-row
  // tiles; each CTA holds half of B, so a slot is 32 KiB at tile_n 256 and
  // deeper rings fit) when at least half a wave of pair tiles exists, then
  // single-CTA 128-row tiles from the widest down.  Half a wave of 256 x 256
  // tiles beats one to two waves of 256 x 128 ones, which run at ~72 % of
  // the wider tiles' rate (2048^3: 20.4 vs 26.5 us; 4096 x 1024 x 8192: 47.7
  // vs 72.3 us).  A candidate must
  // fit the shared-memory budget; single-CTA widths narrow while the widest
  // leaves most SMs idle (fewer tiles than SMs).
  // Ring depth actually built: a pipelined plan whose K has fewer slices than
  // `stages` (and too few for any K split) gets one slot per slice; the
  // extra slots would only take shared memory (256^3, 4 slices: 8.2 us with
  // 4 slots against 9.8 us with 6, L2 flushed).
  const int64_t k_slices = cdiv(K, kBK);
  const int ring_stages =
      (variant == GEMM_PIPELINED && want_split == 0 && k_slices >= 1 && k_slices < 16)
          ? static_cast<int>(std::min<int64_t>(stages, k_slices))
          : stages;
  struct Cand { int cg, bn; };
  const Cand cands[5] = {{2, 256}, {2, 128}, {1, 256}, {1, 128}, {1, 64}};
  int chosen = 0, chosen_cg = 1, chosen_bufs = 0, chosen_clusters = 0, chosen_groups = 1;
  size_t chosen_smem = 0;
  for (int i = 0; i < 5; ++i) {
    const int cg = cands[i].cg, bn = cands[i].bn;
    if (want_bn != 0 && bn != want_bn) continue;
    if (want_cg != 0 && cg != want_cg) continue;
    // Eight epilogue warps where the epilogue is not hidden behind the main
    // loop: short K, a single row of tiles (8192 x 8192 x 512: 59.7 ->
    // 55.3 us; 16896 x 512 x 640 13.3 -> 13.0 us), or a C whose rows are not
    // 16-byte multiples, which is stored row by row instead of by the copy
    // engine (4095 x 4097 x 8191: 241.1 -> 235.4 us).  Elsewhere four: a
    // second epilogue warp on the MMA issuer's sub-partition cost 0.9 % of
    // the cycles at 8192^3.
    const bool rowwise_c = (N * ((tuning && tuning->out_f32) ? 4 : 2)) % 16 != 0;
    const int groups =
        (tuning && tuning->epi_groups) ? tuning->epi_groups
                                       : ((cdiv(K, kBK) <= 16 || cdiv(std::max<int64_t>(M, 1), kBM * cg) == 1 ||
                                           rowwise_c)
                                              ? 2
                                              : 1);
    int bufs = 2;
    const int a_rows = ring_a_rows(cg, M);
    size_t need = kernel_smem_bytes(bn, ring_stages, bufs, cg, groups, a_rows);
    if (need > static_cast<size_t>(dev.smem_optin)) {
      bufs = 1;
      need = kernel_smem_bytes(bn, ring_stages, bufs, cg, groups, a_rows);
    }
    if (need > static_cast<size_t>(dev.smem_optin)) continue;
    const int64_t tiles =
        cdiv(std::max<int64_t>(M, 1), kBM * cg) * cdiv(std::max<int64_t>(N, 1), bn);
    int clusters = 0;
    if (cg == 2) {
      // Auto mode takes pairs only for problems with at least half a wave of pair tiles.
      if (want_cg == 0 && M <= kBM) continue;
      const gemm_status_t cq = pair_clusters(ctx, bn, need, &clusters);
      if (cq != GEMM_OK) return cq;
      if (clusters < 1) continue;
      if (want_cg == 0 && 2 * tiles < clusters) continue;
    }
    chosen = bn;
    chosen_cg = cg;
    chosen_smem = need;
    chosen_bufs = bufs;
    chosen_groups = groups;
    chosen_clusters = clusters;
    // Whole tiles that keep at least 80 % of the SMs busy are wide enough:
    // 128 x 16384 x 2048 runs 20.5 us on 128 tiles 128 wide, 26.1 us on 256
    // tiles 64 wide.
    if (want_bn != 0 || cg == 2 || 10 * tiles >= 8 * static_cast<int64_t>(dev.sm_count))
      break;
    // Few tiles: a width whose tiles can be split in two along K (see below)
    // and then keep at least 80 % of the SMs busy is wide enough.
    if (cg == 1 && variant == GEMM_PIPELINED && want_split != -1 &&
        2 * tiles <= dev.sm_count && 10 * 2 * tiles >= 8 * dev.sm_count &&
        cdiv(K, kBK) >= 16 && cdiv(K, kBK) % 2 == 0 &&
        static_cast<int64_t>(ring_stages) *
                (static_cast<int64_t>(ring_a_rows(cg, M)) * kBK * 2 + static_cast<int64_t>(bn) * kBK * 2) >=
            static_cast<int64_t>(epi_cta_partial_bytes(bn, groups)))
      break;
  }
  if (chosen == 0) {
    return fail(GEMM_ERR_SMEM_BUDGET,
                "stages=%d does not fit %d B of shared memory at tile width %d (ring %zu B)",
                stages, dev.smem_optin, want_bn ? want_bn : 64,
                gemm_smem_bytes(kBM, want_bn ? want_bn : 64, kBK, 2, stages));
  }

  p->M = M;
  p->N = N;
  p->K = K;
  p->dtype = dtype;
  p->epi = epi;
  p->stages = stages;
  p->ring_stages = ring_stages;
  p->variant = variant;
  p->sm_count = dev.sm_count;
  p->timeout_ns = w.timeout;
  p->num_acc = variant == GEMM_SINGLE_BUFFER ? 1 : 2;
  p->max_ctas = want_ctas;
  p->debug_fault = tuning ? tuning->debug_fault : 0;
  p->out_f32 = tuning ? tuning->out_f32 : 0;
  p->b_kn = tuning ? tuning->b_kn : 0;
  p->bn = chosen;
  p->cg = chosen_cg;
  p->smem = chosen_smem;
  p->store_bufs = chosen_bufs;
  p->epi_groups = chosen_groups;
  p->tiles_m = cdiv(M, kBM * chosen_cg);
  p->tiles_n = cdiv(N, chosen);
  p->num_tiles = p->tiles_m * p->tiles_n;
  if (p->num_tiles > kMaxDim) {
    return fail(GEMM_ERR_INVALID_ARG, "too many output tiles");
  }
  p->raster_group = want_group > 0 ? want_group : (chosen_cg == 2 ? 8 : 16);
  if (p->tiles_m > 0)
    p->raster_group = static_cast<int>(std::min<int64_t>(p->raster_group, p->tiles_m));
  // Walkers: persistent CTAs (or CTA pairs) that can be resident at once.
  int walkers;
  if (chosen_cg == 2) {
    walkers = chosen_clusters;
    if (want_ctas > 0) walkers = std::min(walkers, std::max(1, want_ctas / 2));
  } else {
    walkers = p->sm_count;
    if (want_ctas > 0) walkers = std::min(walkers, want_ctas);
  }
  // The last, partial wave.  Stream-K: leave (full waves - 1) waves of
  // whole tiles and share the K iterations of the remaining one to two
  // waves' tiles evenly among all walkers; each walker then holds at least
  // one tile's worth, so a tile is split between at most two walkers and the
  // owner (holding K slice 0, processed last) adds one partial.  The owner
  // stages that partial in its idle ring, which must hold 4 x 32 x BN fp32.
  // Narrow tiles: cut the leftover tiles along N (>= 64 columns each); no
  // reduction, but narrow MMAs re-read A for fewer columns, so automatic
  // mode uses them only when stream-K does not apply and the wave is at
  // most a quarter full.
  const int64_t k_blocks = cdiv(K, kBK);
  // CTA pairs, and single CTAs streaming B (one row of tiles), with an even
  // ring of >= 6 slices group the slices in pairs: stages / 2 slots of two K
  // slices each, the same shared memory, but one barrier round trip per 8
  // MMAs instead of 4 (measured +2-5 % on pairs) and each B row read in
  // 256-byte runs (+8-21 % on 64-128-row problems).  Two slots (4 slices)
  // are too shallow: 8192^3 drops from 1647 to 1498 TFLOP/s.
  p->k_sub = ((chosen_cg == 2 || p->tiles_m == 1) && variant == GEMM_PIPELINED &&
              ring_stages % 2 == 0 && ring_stages >= 6 && k_blocks >= 4)
                 ? 2
                 : 1;
  const int64_t k_slots = cdiv(K, kBK * p->k_sub);
  p->dp_tiles = p->num_tiles;
  p->tail_splits = 1;
  p->sk_tiles = 0;
  const int64_t slice_a = static_cast<int64_t>(ring_a_rows(chosen_cg, M)) * kBK * 2;
  const int64_t ring_all = static_cast<int64_t>(ring_stages) *
                           (slice_a + static_cast<int64_t>(p->bn / chosen_cg) * kBK * 2);
  const bool ring_holds_partial =
      ring_all >= static_cast<int64_t>(epi_cta_partial_bytes(p->bn, p->epi_groups));
  if (variant == GEMM_PIPELINED && want_split == 0 && chosen_cg == 1 && p->num_tiles > 0 &&
      2 * p->num_tiles <= walkers && k_blocks >= 16 && k_blocks % 2 == 0 && ring_holds_partial) {
    // Few tiles (at most half a wave): split every tile in two equal K halves
    // on two walkers -- the stream-K machinery with sk_tiles = tiles and
    // exactly two walkers per tile (first half owns, second contributes).
    p->dp_tiles = 0;
    p->sk_tiles = p->num_tiles;
    walkers = static_cast<int>(2 * p->num_tiles);
    // Walkers 2t (first half, owner) and 2t + 1 (second half) are adjacent
    // CTAs: launched as 2-CTA clusters, the partial goes through distributed
    // shared memory instead of a workspace round trip through L2.
    p->sk_cluster = 1;
  } else if (variant == GEMM_PIPELINED && want_split != -1 && p->num_tiles > 0) {
    const int64_t rem = p->num_tiles % walkers;
    const int64_t ring = static_cast<int64_t>(ring_stages) *
                         (slice_a + static_cast<int64_t>(p->bn / chosen_cg) * kBK * 2);
    const bool sk_fits = ring >= static_cast<int64_t>(epi_cta_partial_bytes(p->bn, p->epi_groups));
    // Automatic stream-K needs long tiles: exchanging one partial costs about
    // as much as a few K slices, so with short K it loses more than the idle
    // part of the last wave (16896 x 512 x 640: 26 us with, 19 us without).
    // It must also have idle time to recover: with a nearly full last wave
    // the exchanges cost more than they save (3072^3, 68 of 76 pair tiles in
    // the last wave, 5 idle slices per walker: 13 % slower with it; 4096^3,
    // 40 idle slices: 4 % faster).
    const bool sk_ok = rem > 0 && p->num_tiles >= walkers && sk_fits &&
                       (want_split == 1 ? k_slots >= 2
                                        : k_blocks >= kStreamKMinKBlocks &&
                                              (walkers - rem) * k_blocks >=
                                                  static_cast<int64_t>(kStreamKMinIdleSlices) * walkers);
    const int max_s = std::min(kMaxTailSplits, p->bn / kStoreCols);
    if (want_split == 1 || (want_split == 0 && sk_ok)) {
      if (!sk_ok && want_split == 1 && rem > 0) {
        return fail(GEMM_ERR_INVALID_ARG,
                    "stream-K needs at least one full wave of tiles and a ring of >= %d B",
                    static_cast<int>(epi_cta_partial_bytes(p->bn, p->epi_groups)));
      }
      if (sk_ok) {
        p->dp_tiles = (p->num_tiles / walkers - 1) * walkers;
        p->sk_tiles = p->num_tiles - p->dp_tiles;
      }
    } else if (rem > 0 && (want_split >= 2 || rem * 4 <= walkers) &&
               !(tuning && tuning->b_kn)) {
      int64_t S = want_split >= 2 ? want_split : std::min<int64_t>(walkers / rem, max_s);
      if (S >= 2 && S <= max_s && p->bn % S == 0) {
        p->dp_tiles = p->num_tiles - rem;
        p->tail_splits = static_cast<int>(S);
      } else if (want_split >= 2) {
        return fail(GEMM_ERR_INVALID_ARG,
                    "tail_split %d does not divide tile width %d into >= %d-column tiles",
                    want_split, p->bn, kStoreCols);
      }
    }
  }
  // One row of tiles streaming a large B (memory-bound): prefetch B into L2
  // in 512-byte row runs, 8 slices ahead.
  p->prefetch_kb = (p->tiles_m == 1 && p->k_sub == 1 && k_blocks >= 4 * kPrefetchSlices &&
                    !(tuning && tuning->b_kn))
                       ? 8
                       : 0;
  // Serpentine K.  One wave of walkers covers raster_group tile rows and
  // about walkers / raster_group tile columns, so it reads (rows + columns)
  // x K operand elements; the next wave reuses its A rows (same raster group)
  // only if they survive in L2 for a whole wave.  When that footprint exceeds
  // half of L2, alternating the K direction makes a wave start on the slices
  // its predecessor read last.  (8192^3: ~73 MB per wave, +1.7 %; 4096^3:
  // ~37 MB, no change.)
  {
    const int want_serp = tuning ? tuning->k_serpentine : 0;
    const int64_t wave_rows = std::min<int64_t>(p->tiles_m, p->raster_group) * kBM * chosen_cg;
    const int64_t wave_cols =
        std::min<int64_t>(p->tiles_n, cdiv(walkers, std::max(1, p->raster_group))) * p->bn;
    const double wave_bytes = static_cast<double>(wave_rows + wave_cols) * static_cast<double>(K) * 2.0;
    const bool auto_on = p->num_tiles > walkers && wave_bytes > 0.5 * static_cast<double>(dev.l2_bytes);
    p->k_serpentine =
        (p->tiles_m > 1 && (want_serp == 1 || (want_serp == 0 && auto_on))) ? 1 : 0;
  }
  // Operands that do not stay in L2 (more than 3/4 of it): each CTA's first
  // slices come from DRAM, so it prefetches them into L2 while the previous
  // kernel finishes (skinny 64 x 8192 x 8192, 135 MB against a 135.5 MB L2:
  // 26.2 -> 25.6 us back to back).  L2-resident operands skip it: the
  // prefetches would only queue ahead of the ring's copies (16896 x 512 x
  // 640: 13.0 -> 13.9 us).
  // Stream-K share first, whole tiles after: the owners' fix-ups then
  // overlap their next tiles instead of ending the launch (GELU layer
  // 3072 x 16384 x 4096 -3.3 %, 4096^3 -1.2 %).  Not with the serpentine K
  // order, whose alternating waves it disturbs (K = 8192 shapes 2-5 %
  // slower), nor for the cluster split, which has no whole tiles.
  p->sk_first = (p->sk_tiles > 0 && !p->sk_cluster && !p->k_serpentine) ? 1 : 0;
  p->l2_prefetch_first = static_cast<double>(M + N) * static_cast<double>(K) * 2.0 >
                                 0.75 * static_cast<double>(dev.l2_bytes)
                             ? 1
                             : 0;
  const int64_t tail = p->num_tiles - p->dp_tiles;
  p->num_units = p->sk_tiles > 0 ? p->dp_tiles : p->dp_tiles + tail * p->tail_splits;
  if (p->num_units > kMaxDim) return fail(GEMM_ERR_INVALID_ARG, "too many work units");
  p->grid = chosen_cg * static_cast<int>(
                           std::min<int64_t>(p->sk_tiles > 0 ? walkers : p->num_units, walkers));
  return GEMM_OK;
}

}  // namespace

gemm_status_t gemm_plan_create_ex(gemm_plan_t** out, int64_t M, int64_t N, int64_t K,
                                  gemm_dtype_t dtype, gemm_epilogue_t epi, int stages,
                                  gemm_variant_t variant, int device,
                                  const gemm_tuning_t* tuning) {
  g_last_error.clear();
  if (!out) return fail(GEMM_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  Wants w;
  gemm_status_t st = check_create_args(M, N, K, dtype, epi, stages, variant, tuning, &w);
  if (st != GEMM_OK) return st;
  if (device < 0) return fail(GEMM_ERR_INVALID_ARG, "device %d < 0", device);
  int ndev = 0;
  cudaError_t e = cudaGetDeviceCount(&ndev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
  if (device >= ndev) return fail(GEMM_ERR_INVALID_ARG, "device %d >= count %d", device, ndev);
  DeviceGuard guard(device);
  if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
  gemm_device_desc_t desc;
  st = device_props(device, &desc);
  if (st != GEMM_OK) return st;

  gemm_plan* p = new (std::nothrow) gemm_plan();
  if (!p) return fail(GEMM_ERR_INVALID_ARG, "out of host memory");
  p->device = device;
  size_t optin = static_cast<size_t>(desc.smem_optin);
  st = plan_layout(p, desc, cuda_pair_clusters, &optin, M, N, K, dtype, epi, stages, variant,
                   tuning, w);
  if (st != GEMM_OK) {
    delete p;
    return st;
  }

  // The limit is per kernel function, shared by every plan on the device:
  // always raise it to the device maximum, never to this plan's own size, so
  // a later plan with a smaller ring cannot lower it under an earlier one.
  e = set_smem(p->bn, p->cg, static_cast<size_t>(desc.smem_optin));
  if (e != cudaSuccess) {
    delete p;
    return cuda_fail(e, "cudaFuncSetAttribute(max dynamic smem)");
  }
  // Device memory: the stream-K workspace and flags, and the status word.
  // On a failure gemm_plan_destroy frees whatever was already allocated.
  if (p->sk_tiles > 0) {
    const size_t nflags = static_cast<size_t>(p->sk_tiles) * p->cg * 4 * p->epi_groups;
    if ((e = cudaMalloc(&p->sk_ws, nflags * epi_warp_partial_bytes(p->bn, p->epi_groups))) !=
            cudaSuccess ||
        (e = cudaMalloc(&p->sk_flags, nflags * sizeof(int))) != cudaSuccess ||
        (e = cudaMemset(p->sk_flags, 0, nflags * sizeof(int))) != cudaSuccess) {
      gemm_plan_destroy(p);
      return cuda_fail(e, "cudaMalloc(stream-K workspace)");
    }
  }
  if ((e = cudaMalloc(&p->d_status, 4 * sizeof(int))) != cudaSuccess ||
      (e = cudaMemset(p->d_status, 0, 4 * sizeof(int))) != cudaSuccess) {
    gemm_plan_destroy(p);
    return cuda_fail(e, "cudaMalloc(status)");
  }
  if (tuning) {
    p->tuning = *tuning;
    p->has_tuning = true;
  }
  *out = p;
  return GEMM_OK;
}

gemm_status_t gemm_plan_create(gemm_plan_t** out, int64_t M, int64_t N, int64_t K,
                               gemm_dtype_t dtype, gemm_epilogue_t epi, int stages,
                               gemm_variant_t variant, int device) {
  return gemm_plan_create_ex(out, M, N, K, dtype, epi, stages, variant, device, nullptr);
}

gemm_status_t gemm_run(gemm_plan_t* plan, const void* A, const void* B, void* C, int64_t M,
                       int64_t N, int64_t K, gemm_dtype_t dtype, gemm_epilogue_t epi, int stages,
                       void* stream_handle) {
  return gemm_run_bias(plan, A, B, nullptr, C, M, N, K, dtype, epi, stages, stream_handle);
}

gemm_status_t gemm_run_bias(gemm_plan_t* plan, const void* A, const void* B, const void* bias,
                            void* C, int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                            gemm_epilogue_t epi, int stages, void* stream_handle) {
  g_last_error.clear();
  if (!plan) return fail(GEMM_ERR_INVALID_ARG, "plan is NULL");
  gemm_status_t st = check_common(M, N, K, dtype, epi, stages);
  if (st != GEMM_OK) return st;
  if (M != plan->M || N != plan->N || K != plan->K || dtype != plan->dtype || epi != plan->epi ||
      stages != plan->stages)
    return fail(GEMM_ERR_PLAN_MISMATCH,
                "run (M=%lld N=%lld K=%lld dtype=%d epi=%d stages=%d) differs from the plan "
                "(M=%lld N=%lld K=%lld dtype=%d epi=%d stages=%d)",
                (long long)M, (long long)N, (long long)K, (int)dtype, (int)epi, stages,
                (long long)plan->M, (long long)plan->N, (long long)plan->K, (int)plan->dtype,
                (int)plan->epi, plan->stages);
  if (M == 0 || N == 0) {
    plan->last_kernels = 0;
    return GEMM_OK;
  }
  if (!C) return fail(GEMM_ERR_INVALID_ARG, "C is NULL");
  if (K > 0 && (!A || !B)) return fail(GEMM_ERR_INVALID_ARG, "A or B is NULL");
  const size_t esC = plan->out_f32 ? 4 : 2;   // bytes per element of C
  const size_t bytesA = static_cast<size_t>(M) * K * 2, bytesB = static_cast<size_t>(N) * K * 2;
  const size_t bytesC = static_cast<size_t>(M) * N * esC;
  const int64_t ldc = plan->ldc ? plan->ldc : N;  // C's row pitch (elements)
  const size_t extentC = (static_cast<size_t>(M - 1) * ldc + N) * esC;
  if (ranges_overlap(C, extentC, A, bytesA) || ranges_overlap(C, extentC, B, bytesB))
    return fail(GEMM_ERR_INVALID_ARG, "C overlaps A or B");
  if (bias && ranges_overlap(C, extentC, bias, static_cast<size_t>(N) * 2))
    return fail(GEMM_ERR_INVALID_ARG, "C overlaps the bias");
  if (((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
        reinterpret_cast<uintptr_t>(bias)) & 1u) ||
      (reinterpret_cast<uintptr_t>(C) & (esC - 1)) != 0)
    return fail(GEMM_ERR_INVALID_ARG, "A, B and the bias must be 2-byte and C %zu-byte aligned",
                esC);

  DeviceGuard guard(plan->device);
  if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_handle);
  // Host-side range for profilers and tracers (a no-op without one attached).
  struct NvtxRange {
    NvtxRange() { nvtxRangePushA("gemm_run"); }
    ~NvtxRange() { nvtxRangePop(); }
  } nvtx_range;

  if (K == 0) {  // empty reduction: C = epi(bias), or 0 (GELU(0) = ReLU(0) = 0)
    if (bias) {
      cudaError_t e = launch_bias_fill(C, M, N, bias, plan->dtype == GEMM_BF16,
                                       static_cast<int>(plan->epi), plan->out_f32 != 0,
                                       plan->sm_count, stream);
      if (e != cudaSuccess) return cuda_fail(e, "bias fill launch");
      plan->last_kernels = 1;
      return GEMM_OK;
    }
    cudaError_t e = cudaMemsetAsync(C, 0, bytesC, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    plan->last_kernels = 0;
    return GEMM_OK;
  }

  // Operands whose pitch or base is not 16-byte aligned go through padded
  // scratch.  B's pitch is K (N x K) or, with b_kn, N (K x N).  A K x N B is
  // read through a 4-D view whose 64-column blocks and 8-row groups must lie
  // inside the array, so it is also staged unless N % 64 == 0 and K % 8 == 0
  // (scratch: pitch rounded up to 64 columns, rows up to a multiple of 8,
  // the extra columns and rows zero).
  const bool padA = (K % 8) != 0 || (reinterpret_cast<uintptr_t>(A) & 15u) != 0;
  const int64_t bcols = plan->b_kn ? N : K;   // B's contiguous extent
  const int64_t brows = plan->b_kn ? K : N;
  const int64_t bcol_mult = plan->b_kn ? 64 : 8;
  const bool padB = (bcols % bcol_mult) != 0 || (plan->b_kn && (K % 8) != 0) ||
                    (reinterpret_cast<uintptr_t>(B) & 15u) != 0;
  const int64_t Kp = (K + 7) / 8 * 8;
  const int64_t Bp_cols = (bcols + bcol_mult - 1) / bcol_mult * bcol_mult;
  const int64_t Bp_rows = plan->b_kn ? Kp : brows;
  const void* effA = A;
  const void* effB = B;
  int kernels = 0;
  if (padA || padB) {
    const size_t need = (padA ? static_cast<size_t>(M) * Kp : 0) +
                        (padB ? static_cast<size_t>(Bp_rows) * Bp_cols : 0);
    const size_t need_bytes = need * 2;
    if (need_bytes > plan->scratch_bytes) {
      if (plan->scratch) {
        cudaError_t e = cudaFree(plan->scratch);
        plan->scratch = nullptr;
        plan->scratch_bytes = 0;
        if (e != cudaSuccess) return cuda_fail(e, "cudaFree(scratch)");
      }
      cudaError_t e = cudaMalloc(&plan->scratch, need_bytes);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(scratch)");
      plan->scratch_bytes = need_bytes;
      plan->mapA_ptr = plan->mapB_ptr = nullptr;
    }
    uint16_t* Ap = padA ? plan->scratch : nullptr;
    uint16_t* Bp = padB ? plan->scratch + (padA ? M * Kp : 0) : nullptr;
    cudaError_t e;
    if (!plan->b_kn) {
      e = launch_pad_operands(static_cast<const uint16_t*>(A), M, Ap,
                              static_cast<const uint16_t*>(B), N, Bp, K, Kp, plan->sm_count,
                              stream);
      if (e != cudaSuccess) return cuda_fail(e, "pad kernel launch");
      ++kernels;
    } else {  // rows of different length: one launch per operand
      if (padA) {
        e = launch_pad_operands(static_cast<const uint16_t*>(A), M, Ap, nullptr, 0, nullptr, K,
                                Kp, plan->sm_count, stream);
        if (e != cudaSuccess) return cuda_fail(e, "pad kernel launch");
        ++kernels;
      }
      if (padB) {
        e = launch_pad_operands(static_cast<const uint16_t*>(B), K, Bp, nullptr, 0, nullptr, N,
                                Bp_cols, plan->sm_count, stream);
        if (e != cudaSuccess) return cuda_fail(e, "pad kernel launch");
        ++kernels;
        if (Bp_rows > K) {  // zero rows up to the next multiple of 8
          e = cudaMemsetAsync(Bp + K * Bp_cols, 0,
                              static_cast<size_t>(Bp_rows - K) * Bp_cols * 2, stream);
          if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(B row padding)");
        }
      }
    }
    if (padA) effA = Ap;
    if (padB) effB = Bp;
  }
  // A's pitch (and, for N x K B, B's): Kp when padded (K % 8 == 0 otherwise,
  // so K == Kp); a K x N B has pitch Bp_cols when padded, else N.
  const int64_t Keff = (padA || (padB && !plan->b_kn)) ? Kp : K;
  const int64_t Beff_cols = plan->b_kn ? (padB ? Bp_cols : N) : Keff;
  const int64_t Beff_rows = plan->b_kn ? (padB ? Bp_rows : K) : N;

  const bool tma_store =
      (static_cast<size_t>(ldc) * esC) % 16 == 0 && (reinterpret_cast<uintptr_t>(C) & 15u) == 0;

  // M <= 64 (single CTA tiles): copy only 64 rows of A per slice.
  const uint32_t a_box_rows = static_cast<uint32_t>(ring_a_rows(plan->cg, M));
  if (plan->mapA_ptr != effA || plan->mapK != Keff) {
    st = encode_2d(&plan->tmA, plan->dtype, effA, Keff, M, Keff, kBK, a_box_rows,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (st != GEMM_OK) return st;
    plan->mapA_ptr = effA;
  }
  if (plan->mapB_ptr != effB || plan->mapK != Keff) {
    if (!plan->b_kn)
      st = encode_2d(&plan->tmB, plan->dtype, effB, Keff, N, Keff, kBK,
                     static_cast<uint32_t>(plan->bn / plan->cg), CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    else
      st = encode_b_kn(&plan->tmB, plan->dtype, effB, Beff_cols, Beff_rows,
                       static_cast<uint32_t>(plan->bn / plan->cg / 64));
    if (st != GEMM_OK) return st;
    if (plan->tail_splits > 1) {
      st = encode_2d(&plan->tmBt, plan->dtype, effB, Keff, N, Keff, kBK,
                     static_cast<uint32_t>(plan->bn / plan->tail_splits / plan->cg),
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
      if (st != GEMM_OK) return st;
    } else {
      plan->tmBt = plan->tmB;
    }
    if (plan->prefetch_kb > 0) {
      st = encode_2d(&plan->tmBp, plan->dtype, effB, Keff, N, Keff, kBK * kPrefetchSlices,
                     static_cast<uint32_t>(plan->bn / plan->cg), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
      if (st != GEMM_OK) return st;
    } else {
      plan->tmBp = plan->tmB;
    }
    plan->mapB_ptr = effB;
  }
  plan->mapK = Keff;
  if (tma_store && plan->mapC_ptr != C) {
    // One 128-byte row of 16-bit (64) or fp32 (32) elements per box row.
    st = plan->out_f32 ? encode_2d_f32(&plan->tmC, C, N, M, ldc, 32, 32)
                       : encode_2d(&plan->tmC, plan->dtype, C, N, M, ldc, kStoreCols, 32,
                                   CU_TENSOR_MAP_L2_PROMOTION_NONE);
    if (st != GEMM_OK) return st;
    plan->mapC_ptr = C;
  }

  Params prm;
  std::memset(&prm, 0, sizeof(prm));
  prm.M = static_cast<int>(M);
  prm.N = static_cast<int>(N);
  prm.K = static_cast<int>(Keff);
  prm.tiles_m = static_cast<int>(plan->tiles_m);
  prm.tiles_n = static_cast<int>(plan->tiles_n);
  prm.num_tiles = static_cast<int>(plan->num_tiles);
  prm.k_blocks = static_cast<int>(cdiv(Keff, kBK * plan->k_sub));
  prm.stages = plan->ring_stages / plan->k_sub;
  prm.k_sub = plan->k_sub;
  prm.num_acc = plan->num_acc;
  int cols = plan->bn * plan->num_acc;
  int pow2 = 32;
  while (pow2 < cols) pow2 <<= 1;
  prm.tmem_cols = pow2;
  prm.raster_group = plan->raster_group;
  prm.store_bufs = plan->store_bufs;
  prm.epi_groups = plan->epi_groups;
  prm.bf16 = plan->dtype == GEMM_BF16 ? 1 : 0;
  prm.epilogue = static_cast<int>(plan->epi);
  prm.out_f32 = plan->out_f32;
  prm.tma_store = tma_store ? 1 : 0;
  prm.idesc = ptx::instr_desc_f16(kBM * plan->cg, plan->bn, plan->dtype == GEMM_BF16,
                                  plan->b_kn != 0);
  prm.C = C;
  prm.ldc = ldc;
  prm.status = plan->d_status;
  prm.timeout_ns = plan->timeout_ns;
  prm.dp_tiles = static_cast<int>(plan->dp_tiles);
  prm.tail_splits = plan->tail_splits;
  prm.num_units = static_cast<int>(plan->num_units);
  prm.idesc_tail = ptx::instr_desc_f16(kBM * plan->cg, plan->bn / plan->tail_splits,
                                       plan->dtype == GEMM_BF16, plan->b_kn != 0);
  // One row of tiles across the whole grid: every CTA reads the same A rows,
  // so stagger where each starts along K.
  prm.k_rotate = (plan->tiles_m == 1 && plan->num_tiles > 1) ? 1 : 0;
  prm.k_serpentine = plan->k_serpentine;
  prm.l2_prefetch_first = plan->l2_prefetch_first;
  prm.sk_cluster = plan->sk_cluster;
  prm.sk_first = plan->sk_first;
  prm.inject_fault = plan->debug_fault;
  prm.prefetch_kb = plan->prefetch_kb;
  prm.a_box_rows = static_cast<int>(a_box_rows);
  prm.b_stream = (plan->tiles_m == 1 && plan->cg == 1) ? 1 : 0;
  prm.b_kn = plan->b_kn;
  prm.sk_tiles = static_cast<int>(plan->sk_tiles);
  prm.sk_ws = plan->sk_ws;
  prm.sk_flags = plan->sk_flags;
  prm.sk_slots = plan->sk_tiles > 0
                     ? static_cast<int>(plan->sk_tiles * plan->cg * 4 * plan->epi_groups)
                     : 0;
  prm.bias = bias;

  cudaError_t e = launch(plan->bn, plan->cg, plan->tmA, plan->tmB, plan->tmBt, plan->tmC,
                         plan->tmBp, prm, plan->grid, plan->smem, stream);
  if (e != cudaSuccess) return cuda_fail(e, "GEMM kernel launch");
  ++kernels;
  plan->last_pads = (padA || padB) ? 1 : 0;
  plan->last_tma_store = tma_store ? 1 : 0;
  plan->last_kernels = kernels;
  return GEMM_OK;
}

// Blocks for gemm_run_host.  Row panels of A (whole tiles of rows); column
// panels -- row panels of B -- only for N x K B and K a multiple of 8, so
// that every block's A and B rows start 16-byte aligned inside the staged
// operands (B stored K x N, or a K that needs padding, keeps whole rows of
// C).  One plan per block shape, writing into the whole C (row pitch N).
static gemm_status_t host_panels_setup(gemm_plan_t* plan) {
  if (plan->panel_rows > 0) return GEMM_OK;
  const int64_t M = plan->M, N = plan->N;
  const int64_t tile_m = static_cast<int64_t>(kBM) * plan->cg;
  int pm = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(kHostPanelsMax, M / kHostPanelMinRows)));
  const int64_t rows = cdiv(cdiv(M, pm), tile_m) * tile_m;
  pm = static_cast<int>(cdiv(M, rows));
  int pn = 1;
  int64_t cols = N;
  if (!plan->b_kn && plan->K % 8 == 0) {
    pn = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(kHostPanelsMax, N / kHostPanelMinRows)));
    cols = cdiv(cdiv(N, pn), 256) * 256;
    pn = static_cast<int>(cdiv(N, cols));
  }
  if (pm * pn < 2) {
    plan->panel_rows = M;
    plan->panel_cols = N;
    plan->num_panels = plan->num_col_panels = 1;
    return GEMM_OK;
  }
  const gemm_tuning_t* t = plan->has_tuning ? &plan->tuning : nullptr;
  const int64_t hs[2] = {rows, M - (pm - 1) * rows};
  const int64_t ws[2] = {cols, N - (pn - 1) * cols};
  for (int lr = 0; lr < 2; ++lr)
    for (int lc = 0; lc < 2; ++lc) {
      if ((lr == 1 && hs[1] == rows) || (lc == 1 && ws[1] == cols)) continue;
      gemm_status_t st = gemm_plan_create_ex(&plan->blk[lr][lc], hs[lr], ws[lc], plan->K,
                                             plan->dtype, plan->epi, plan->stages, plan->variant,
                                             plan->device, t);
      if (st != GEMM_OK) return st;
      plan->blk[lr][lc]->ldc = N;
    }
  cudaError_t e = cudaStreamCreateWithFlags(&plan->copy_in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&plan->copy_out, cudaStreamNonBlocking);
  for (cudaEvent_t* ev : {&plan->ev_start, &plan->ev_done})
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  for (int i = 0; i < pm && e == cudaSuccess; ++i)
    e = cudaEventCreateWithFlags(&plan->ev_a[i], cudaEventDisableTiming);
  for (int j = 0; j < pn && e == cudaSuccess; ++j)
    e = cudaEventCreateWithFlags(&plan->ev_b[j], cudaEventDisableTiming);
  for (int b = 0; b < pm * pn && e == cudaSuccess; ++b)
    e = cudaEventCreateWithFlags(&plan->ev_c[b], cudaEventDisableTiming);
  if (e != cudaSuccess) return cuda_fail(e, "streams/events for gemm_run_host");
  plan->panel_rows = rows;
  plan->panel_cols = cols;
  plan->num_panels = pm;
  plan->num_col_panels = pn;
  return GEMM_OK;
}

gemm_status_t gemm_run_host(gemm_plan_t* plan, const void* hA, const void* hB, void* hC,
                            int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                            gemm_epilogue_t epi, int stages, void* stream_handle) {
  g_last_error.clear();
  if (!plan) return fail(GEMM_ERR_INVALID_ARG, "plan is NULL");
  gemm_status_t st = check_common(M, N, K, dtype, epi, stages);
  if (st != GEMM_OK) return st;
  if (M != plan->M || N != plan->N || K != plan->K || dtype != plan->dtype || epi != plan->epi ||
      stages != plan->stages)
    return fail(GEMM_ERR_PLAN_MISMATCH, "run arguments differ from the plan");
  const size_t esC = plan->out_f32 ? 4 : 2;
  const size_t bytesA = static_cast<size_t>(M) * K * 2, bytesB = static_cast<size_t>(N) * K * 2;
  const size_t bytesC = static_cast<size_t>(M) * N * esC;
  if (bytesC == 0) return GEMM_OK;
  if (!hC || (bytesA && !hA) || (bytesB && !hB))
    return fail(GEMM_ERR_INVALID_ARG, "NULL host buffer");
  DeviceGuard guard(plan->device);
  if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_handle);
  cudaError_t e;
  if (!plan->hC) {
    if (bytesA && (e = cudaMalloc(&plan->hA, bytesA)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(A)");
    if (bytesB && (e = cudaMalloc(&plan->hB, bytesB)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(B)");
    if ((e = cudaMalloc(&plan->hC, bytesC)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(C)");
  }
  const bool pipelined = K > 0 && bytesA + bytesB + bytesC >= kHostPanelMinBytes;
  if (pipelined) {
    st = host_panels_setup(plan);
    if (st != GEMM_OK) return st;
  }
  if (!pipelined || plan->num_panels * plan->num_col_panels < 2) {
    if (bytesA && (e = cudaMemcpyAsync(plan->hA, hA, bytesA, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
      return cuda_fail(e, "copy A to device");
    if (bytesB && (e = cudaMemcpyAsync(plan->hB, hB, bytesB, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
      return cuda_fail(e, "copy B to device");
    st = gemm_run(plan, plan->hA, plan->hB, plan->hC, M, N, K, dtype, epi, stages, stream_handle);
    if (st != GEMM_OK) return st;
    if ((e = cudaMemcpyAsync(hC, plan->hC, bytesC, cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
      return cuda_fail(e, "copy C to host");
    if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    return GEMM_OK;
  }

  // Pipelined, in blocks of C.  The host link carries ~200 GB/s each way and
  // ~280 GB/s both ways together, so the copies set the pace: A's row panels
  // and B's row panels (C's column panels) go in on one stream, alternating
  // (A0, B0, A1, B1, ...), so that block (i, j) can start as soon as both of
  // its panels are in; blocks run on the caller's stream as their panels
  // arrive, and each block of C goes back (a 2-D copy) on a second stream
  // while the next ones compute.  (8192^3 fp16: 1.89 ms per call with whole
  // rows of C and B first, ~1.7 ms with 4 x 4 blocks.)
  const int Pm = plan->num_panels, Pn = plan->num_col_panels;
  const int64_t R = plan->panel_rows, Cw = plan->panel_cols;
  auto ck = [&](cudaError_t err, const char* what) -> bool {
    if (err != cudaSuccess) {
      cuda_fail(err, what);
      return false;
    }
    return true;
  };
  const char* hAb = static_cast<const char*>(hA);
  const char* hBb = static_cast<const char*>(hB);
  char* hCb = static_cast<char*>(hC);
  char* dA = static_cast<char*>(plan->hA);
  char* dB = static_cast<char*>(plan->hB);
  char* dC = static_cast<char*>(plan->hC);
  if (!ck(cudaEventRecord(plan->ev_start, stream), "record start") ||
      !ck(cudaStreamWaitEvent(plan->copy_in, plan->ev_start, 0), "copy stream wait") ||
      !ck(cudaStreamWaitEvent(plan->copy_out, plan->ev_start, 0), "copy-out wait"))
    return GEMM_ERR_CUDA;
  int na = 0, nb = 0;
  bool done[kHostPanelsMax][kHostPanelsMax] = {};
  while (na < Pm || nb < Pn) {
    // The next panel in: A while it has no more panels in than B (or B is
    // all in), else B.
    const bool take_a = na < Pm && (na <= nb || nb == Pn);
    if (take_a) {
      const int64_t rows = std::min<int64_t>(R, M - na * R);
      const size_t off = static_cast<size_t>(na) * R * K * 2, len = static_cast<size_t>(rows) * K * 2;
      if (!ck(cudaMemcpyAsync(dA + off, hAb + off, len, cudaMemcpyHostToDevice, plan->copy_in),
              "copy A panel") ||
          !ck(cudaEventRecord(plan->ev_a[na], plan->copy_in), "record A panel"))
        return GEMM_ERR_CUDA;
      ++na;
    } else {
      // One panel of B rows (N x K B), or all of B when it is the only one.
      size_t off = 0, len = bytesB;
      if (Pn > 1) {
        off = static_cast<size_t>(nb) * Cw * K * 2;
        len = static_cast<size_t>(std::min<int64_t>(Cw, N - nb * Cw)) * K * 2;
      }
      if (len && !ck(cudaMemcpyAsync(dB + off, hBb + off, len, cudaMemcpyHostToDevice, plan->copy_in),
                     "copy B panel"))
        return GEMM_ERR_CUDA;
      if (!ck(cudaEventRecord(plan->ev_b[nb], plan->copy_in), "record B panel")) return GEMM_ERR_CUDA;
      ++nb;
    }
    // Every block whose two panels are now in.
    for (int i = 0; i < na; ++i)
      for (int j = 0; j < nb; ++j) {
        if (done[i][j]) continue;
        done[i][j] = true;
        const int64_t rows = std::min<int64_t>(R, M - i * R), cols = std::min<int64_t>(Cw, N - j * Cw);
        gemm_plan* bp = plan->blk[rows == R ? 0 : 1][cols == Cw ? 0 : 1];
        const size_t c_off = (static_cast<size_t>(i) * R * N + static_cast<size_t>(j) * Cw) * esC;
        const size_t b_off = plan->b_kn ? 0 : static_cast<size_t>(j) * Cw * K * 2;
        if (!ck(cudaStreamWaitEvent(stream, plan->ev_a[i], 0), "wait A panel") ||
            !ck(cudaStreamWaitEvent(stream, plan->ev_b[j], 0), "wait B panel"))
          return GEMM_ERR_CUDA;
        st = gemm_run(bp, dA + static_cast<size_t>(i) * R * K * 2, dB + b_off, dC + c_off, rows, cols,
                      K, dtype, epi, stages, stream_handle);
        if (st != GEMM_OK) return st;
        cudaEvent_t ev = plan->ev_c[i * Pn + j];
        if (!ck(cudaEventRecord(ev, stream), "record C block") ||
            !ck(cudaStreamWaitEvent(plan->copy_out, ev, 0), "copy-out wait") ||
            !ck(cudaMemcpy2DAsync(hCb + c_off, static_cast<size_t>(N) * esC, dC + c_off,
                                  static_cast<size_t>(N) * esC, static_cast<size_t>(cols) * esC, rows,
                                  cudaMemcpyDeviceToHost, plan->copy_out),
                "copy C block to host"))
          return GEMM_ERR_CUDA;
      }
  }
  if (!ck(cudaEventRecord(plan->ev_done, plan->copy_out), "record done") ||
      !ck(cudaStreamWaitEvent(stream, plan->ev_done, 0), "wait done") ||
      !ck(cudaStreamSynchronize(stream), "cudaStreamSynchronize"))
    return GEMM_ERR_CUDA;
  return GEMM_OK;
}

gemm_status_t gemm_plan_check(gemm_plan_t* plan, int32_t* device_status, int32_t* detail) {
  g_last_error.clear();
  if (!plan || !device_status) return fail(GEMM_ERR_INVALID_ARG, "NULL argument");
  DeviceGuard guard(plan->device);
  if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  int h[4] = {0, 0, 0, 0};
  e = cudaMemcpy(h, plan->d_status, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read status word");
  e = cudaMemset(plan->d_status, 0, sizeof(h));
  if (e != cudaSuccess) return cuda_fail(e, "clear status word");
  if (h[0] != 0 && plan->sk_flags) {
    // A launch that gave up part-way may have left partial-ready flags raised.
    e = cudaMemset(plan->sk_flags, 0,
                   static_cast<size_t>(plan->sk_tiles) * plan->cg * 4 * plan->epi_groups *
                       sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clear stream-K flags");
  }
  *device_status = h[0];
  if (detail) *detail = h[1];
  // Block plans of gemm_run_host keep status words of their own.
  gemm_plan* panels[4] = {plan->blk[0][0], plan->blk[0][1], plan->blk[1][0], plan->blk[1][1]};
  for (gemm_plan* pp : panels) {
    if (!pp) continue;
    int32_t ds = 0, dd = 0;
    gemm_status_t st = gemm_plan_check(pp, &ds, &dd);
    if (st != GEMM_OK) return st;
    if (*device_status == 0 && ds != 0) {
      *device_status = ds;
      if (detail) *detail = dd;
    }
  }
  return GEMM_OK;
}

namespace {

void fill_info(const gemm_plan* plan, gemm_plan_info_t* info) {
  info->tile_m = kBM * plan->cg;
  info->tile_n = plan->bn;
  info->tile_k = kBK;
  info->stages = plan->ring_stages;
  info->accumulators = plan->num_acc;
  info->raster_group = plan->raster_group;
  info->grid = plan->grid;
  info->num_tiles = plan->num_tiles;
  info->smem_bytes = plan->smem;
  info->pads_operands = plan->last_pads;
  info->tma_store = plan->last_tma_store;
  info->kernels_per_run = plan->last_kernels;
  info->sm_count = plan->sm_count;
  info->k_serpentine = plan->k_serpentine;
  info->epi_groups = plan->epi_groups;
  info->l2_prefetch_first = plan->l2_prefetch_first;
  info->sk_cluster = plan->sk_cluster;
  info->cta_group = plan->cg;
  info->tail_tiles = plan->num_tiles - plan->dp_tiles;
  info->tail_splits = plan->tail_splits;
  info->work_units = plan->num_units;
  info->stream_k = plan->sk_tiles > 0 ? 1 : 0;
  info->out_f32 = plan->out_f32;
  info->b_kn = plan->b_kn;
  info->k_sub = plan->k_sub;
  info->host_panels =
      plan->num_panels * plan->num_col_panels >= 2 ? plan->num_panels * plan->num_col_panels : 0;
  info->stream_k_first = plan->sk_first;
  if (plan->sk_tiles > 0) info->tail_tiles = plan->sk_tiles;
}

}  // namespace

gemm_status_t gemm_plan_get_info(const gemm_plan_t* plan, gemm_plan_info_t* info) {
  if (!plan || !info) return fail(GEMM_ERR_INVALID_ARG, "NULL argument");
  fill_info(plan, info);
  return GEMM_OK;
}

gemm_status_t gemm_device_query(int device, gemm_device_desc_t* desc) {
  g_last_error.clear();
  if (!desc) return fail(GEMM_ERR_INVALID_ARG, "desc is NULL");
  if (device < 0) return fail(GEMM_ERR_INVALID_ARG, "device %d < 0", device);
  int ndev = 0;
  cudaError_t e = cudaGetDeviceCount(&ndev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
  if (device >= ndev) return fail(GEMM_ERR_INVALID_ARG, "device %d >= count %d", device, ndev);
  DeviceGuard guard(device);
  if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
  gemm_device_desc_t d;
  gemm_status_t st = device_props(device, &d);
  if (st != GEMM_OK) return st;
  // Any pair instance at one CTA per SM gives the count: the 256-wide tile's
  // six-slice ring with four epilogue warps.
  size_t optin = static_cast<size_t>(d.smem_optin);
  const size_t smem = kernel_smem_bytes(256, 6, 2, 2, 1);
  if (smem > optin) return fail(GEMM_ERR_UNSUPPORTED, "no pair instance fits %zu B", optin);
  st = cuda_pair_clusters(&optin, 256, smem, &d.pair_clusters);
  if (st != GEMM_OK) return st;
  *desc = d;
  return GEMM_OK;
}

gemm_status_t gemm_plan_describe(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                                 gemm_epilogue_t epi, int stages, gemm_variant_t variant,
                                 const gemm_tuning_t* tuning, const gemm_device_desc_t* desc,
                                 gemm_plan_info_t* info) {
  g_last_error.clear();
  if (!desc || !info) return fail(GEMM_ERR_INVALID_ARG, "NULL argument");
  if (desc->sm_count < 1 || desc->smem_optin < 1 || desc->l2_bytes < 0 ||
      desc->pair_clusters < 0)
    return fail(GEMM_ERR_INVALID_ARG,
                "device description out of range (sm_count %d, smem_optin %d, l2_bytes %lld, "
                "pair_clusters %d)",
                desc->sm_count, desc->smem_optin, static_cast<long long>(desc->l2_bytes),
                desc->pair_clusters);
  Wants w;
  gemm_status_t st = check_create_args(M, N, K, dtype, epi, stages, variant, tuning, &w);
  if (st != GEMM_OK) return st;
  gemm_plan p;  // host fields only: nothing is allocated for it
  st = plan_layout(&p, *desc, desc_pair_clusters, const_cast<gemm_device_desc_t*>(desc), M, N, K,
                   dtype, epi, stages, variant, tuning, w);
  if (st != GEMM_OK) return st;
  fill_info(&p, info);
  return GEMM_OK;
}

void gemm_plan_destroy(gemm_plan_t* plan) {
  if (!plan) return;
  {
    DeviceGuard guard(plan->device);
    if (guard.err == cudaSuccess) {
      cudaDeviceSynchronize();
      if (plan->d_status) cudaFree(plan->d_status);
      if (plan->sk_ws) cudaFree(plan->sk_ws);
      if (plan->sk_flags) cudaFree(plan->sk_flags);
      if (plan->scratch) cudaFree(plan->scratch);
      if (plan->hA) cudaFree(plan->hA);
      if (plan->hB) cudaFree(plan->hB);
      if (plan->hC) cudaFree(plan->hC);
      for (cudaStream_t cs : {plan->copy_in, plan->copy_out})
        if (cs) cudaStreamDestroy(cs);
      for (cudaEvent_t ev : {plan->ev_start, plan->ev_done})
        if (ev) cudaEventDestroy(ev);
      for (int i = 0; i < kHostPanelsMax; ++i) {
        if (plan->ev_a[i]) cudaEventDestroy(plan->ev_a[i]);
        if (plan->ev_b[i]) cudaEventDestroy(plan->ev_b[i]);
      }
      for (cudaEvent_t ev : plan->ev_c)
        if (ev) cudaEventDestroy(ev);
    }
  }
  for (auto& row : plan->blk)
    for (gemm_plan* bp : row) gemm_plan_destroy(bp);
  delete plan;
}

}  // extern "C"
