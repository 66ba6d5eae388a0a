// kernel_params.h -- launch parameters and compile-time geometry shared by
// the host planner (gemm_api.cu) and the device kernels.
#pragma once

#include <cstddef>
#include <cstdint>

// 1 in the bounds-checked build (device-side range checks that record
// GEMM_ERR_BOUNDS instead of making the access), 0 in the normal build.
#ifndef SPGEMM_BOUNDS_CHECKS
#define SPGEMM_BOUNDS_CHECKS 0
#endif

namespace spgemm {

constexpr int kBM = 128;          // CTA tile rows (one TMEM lane per row)
constexpr int kBK = 64;           // K slice: 64 x 16-bit = one 128-byte swizzle row
constexpr int kUmmaK = 16;        // K of one tcgen05.mma kind::f16
// Epilogue warps: one or two per TMEM lane quarter (a warp may read only the
// quarter warp % 4), each taking one column group of the tile; a kernel
// instance has one group (warps 2-5) or two (warps 2-9), Params::epi_groups.
constexpr int kEpiColGroups = 2;                 // at most
constexpr int kEpiWarps = 4 * kEpiColGroups;     // at most
// Threads of a CTA: warp 0 TMA producer, warp 1 MMA issuer, 4 x groups epilogue.
__host__ __device__ constexpr int kernel_threads(int epi_groups) { return 64 + 128 * epi_groups; }
constexpr int kMaxStages = 8;
constexpr uint32_t kStageA = kBM * kBK * 2;             // 16 KiB
constexpr int kStoreCols = 64;                          // epilogue step: 64 columns
constexpr uint32_t kStoreBuf = 32u * kStoreCols * 2u;   // 32 rows x 128 B = 4 KiB
constexpr uint32_t kBarrierBytes = 8u * (2 * kMaxStages + 5 + 2 * kEpiWarps) + 16u;
constexpr uint32_t kAlignSlack = 1024u;

constexpr int kStatusTimeout = 6;  // == GEMM_ERR_TIMEOUT
constexpr int kStatusBounds = 7;   // == GEMM_ERR_BOUNDS (bounds-checked build)

constexpr int kMaxTailSplits = 4;     // narrow tiles a tail tile may be cut into (N >= 64 each)
constexpr int kPrefetchSlices = 4;    // K slices per L2 prefetch box (4 x 128 B per row)
constexpr int kStreamKMinKBlocks = 32;  // automatic stream-K only for K >= 32 slices

// Where a device-side wait ran out (status word [1]): role << 16 | wait id.
constexpr int kDetailProducerEmpty = (1 << 16) | 1;
constexpr int kDetailProducerDrain = (1 << 16) | 2;
constexpr int kDetailMmaAccEmpty = (2 << 16) | 1;
constexpr int kDetailMmaFull = (2 << 16) | 2;
constexpr int kDetailMmaDrain = (2 << 16) | 3;
constexpr int kDetailEpiFull = (3 << 16) | 1;
constexpr int kDetailSkFlag = (3 << 16) | 2;
constexpr int kDetailSkCopy = (3 << 16) | 3;
constexpr int kDetailSkFree = (3 << 16) | 4;
// Which range check failed (status word [1] with kStatusBounds): role << 16 |
// 16 + check id (the bounds-checked build only).
constexpr int kCheckSmemLayout = (0 << 16) | 16;  // ring + staging + barriers exceed the launch's smem
constexpr int kCheckTile = (1 << 16) | 16;        // unit's tile index or tile coordinates
constexpr int kCheckKSlice = (1 << 16) | 17;      // K slot outside the unit's range or the K extent
constexpr int kCheckTmaCoord = (1 << 16) | 18;    // copy coordinate out of range or not 16-byte aligned
constexpr int kCheckMmaTmem = (2 << 16) | 16;     // accumulator columns beyond the TMEM allocation
constexpr int kCheckMmaSlot = (2 << 16) | 17;     // ring slot index beyond the ring
constexpr int kCheckEpiTmem = (3 << 16) | 16;     // TMEM columns read beyond the allocation
constexpr int kCheckStaging = (3 << 16) | 17;     // staging buffer beyond the warp's staging area
constexpr int kCheckStore = (3 << 16) | 18;       // C store outside the tile grid or unaligned
constexpr int kCheckPartial = (3 << 16) | 19;     // stream-K partial / flag index beyond the workspace
constexpr int kCheckFixup = (3 << 16) | 20;       // partial's shared-memory region beyond the ring

struct Params {
  int M, N;              // output extent
  int K;                 // reduction length seen by the tensor maps (padded when staged)
  int tiles_m, tiles_n;
  int num_tiles;
  int k_blocks;          // ceil(K / (kBK * k_sub)): ring slots of K per tile
  int stages;            // ring depth in slots, 1..kMaxStages
  int num_acc;           // TMEM accumulators, 1 or 2
  int tmem_cols;         // allocated TMEM columns (power of two >= 32)
  int raster_group;      // tile rows per raster group
  int store_bufs;        // staging buffers per active epilogue warp (1 or 2)
  int epi_groups;        // epilogue column groups: 1 (warps 2-5) or 2 (warps 2-9)
  int bf16;              // element type: 0 fp16, 1 bf16
  int epilogue;          // 0 none, 1 tanh-GELU, 2 ReLU
  int out_f32;           // C element type: 0 = the input type, 1 = fp32
  int tma_store;         // 1: bulk tensor stores of C; 0: masked st.global
  uint32_t idesc;        // tcgen05.mma instruction descriptor
  void* C;               // used by the st.global path
  int64_t ldc;
  int* status;           // device status word: [0] code, [1] detail
  unsigned long long timeout_ns;
  // Work units: tiles [0, dp_tiles) run whole; each remaining ("tail") tile
  // is cut along N into tail_splits narrower tiles of BN / tail_splits
  // columns, so the last, partial wave keeps more CTAs busy for a shorter
  // time.  num_units = dp_tiles + tail tiles * tail_splits.  Narrow tiles use
  // the B tensor map with the smaller box and the MMA descriptor idesc_tail.
  int dp_tiles;
  int tail_splits;
  int num_units;
  uint32_t idesc_tail;
  // Stream-K (sk_tiles > 0): after the dp_tiles whole tiles, the remaining
  // sk_tiles * k_blocks K iterations are shared out in contiguous ranges, one
  // per walker (at least one tile's worth each, so a tile spans at most two
  // walkers).  The walker holding a tile's first K slices owns it: the other
  // writes its fp32 partial to sk_ws and raises sk_flags; the owner adds it
  // and stores.  Mutually exclusive with tail_splits > 1.
  int sk_tiles;
  float* sk_ws;
  int* sk_flags;
  // 1: each walker takes its stream-K share first and its whole tiles after
  // (the stream-K tiles are then tiles [0, sk_tiles) and the whole ones
  // follow).  A contributor's piece is the first of its share, so its
  // partial is published early; the owner's fix-up reads it from L2 and
  // overlaps the walker's next tile instead of ending the launch.  0: whole
  // tiles first, stream-K tiles [dp_tiles, num_tiles) last, the owner staging
  // the partial in its then idle ring.
  int sk_first;
  int sk_slots;          // epilogue-warp partials (and flags) sk_ws / sk_flags hold
  // 1: each unit starts its K loop at a different slice (wrapping around),
  // so CTAs that share the same A rows do not all read the same A slice at
  // the same time (used when a single row of tiles spans the whole grid).
  int k_rotate;
  // 1: a walker's odd-numbered units (x.seq odd) load their K slices in
  // descending order, so each wave of tiles begins on the slices the previous
  // wave read last, which are the ones most likely still in L2.  Only the
  // copy order changes: the MMA loop counts iterations, not slice indexes.
  int k_serpentine;
  // 1: before waiting on the previous kernel, the producer prefetches into L2
  // the slices its ring will hold first (operands above 3/4 of L2, whose
  // first slices come from DRAM; for L2-resident operands the prefetches
  // only delay the ring's own copies).
  int l2_prefetch_first;
  // 1: every tile is split into two K halves whose walkers form a cluster of
  // two CTAs (owner = rank 0, contributor = rank 1).  The partial goes
  // through distributed shared memory instead of the workspace: once the
  // owner's MMAs are done it tells the contributor that its ring is free,
  // and the contributor bulk-copies the partial (staged in its own idle
  // ring) into that ring.
  int sk_cluster;
  // > 0: the producer also prefetches B into L2, prefetch_kb slices ahead,
  // through a tensor map whose box spans 4 K slices (512 contiguous bytes of
  // each row): memory-bound shapes then read B in longer runs.
  int prefetch_kb;
  // 1: every element of B is read by one CTA only (a single row of
  // single-CTA tiles), so B's copies carry an evict-first L2 policy.
  int b_stream;
  // Rows of the A box the copy engine writes per CTA (128, or 64 when M <= 64:
  // the other 64 rows of the slot are left as they are -- they only feed
  // output rows >= M, which are never stored).
  int a_box_rows;
  // 1: B is stored K x N (N contiguous) and read MN-major.  The B map is 4-D,
  // (64 columns, 8 K rows, 64-column blocks, groups of 8 K rows), so one box
  // lands in shared memory as 1024-byte swizzle atoms ordered [K group]
  // [column block]: the blocks of one K group side by side.
  int b_kn;
  // 64-wide K slices per ring slot (1 or 2); stages and k_blocks count slots.
  int k_sub;
  // Per-column bias (N values of the input type), added to the fp32
  // accumulator before the epilogue function; nullptr for none.
  const void* bias;
  // Test hook: 1 = the producer of CTA 0 announces but never issues the
  // copies of its first K slice; 2 = (bounds-checked build) the range check
  // of that copy is made to fail, the coordinates themselves being valid
  // (see gemm_tuning_t::debug_fault).
  int inject_fault;
};

// Columns of one epilogue column group for a unit `n_width` columns wide:
// all of it with one group; with two, half of it, but whole 64-column store
// chunks (a 64-wide unit then has one non-empty group).
__host__ __device__ constexpr int epi_group_cols(int n_width, int groups) {
  return groups < 2 ? n_width
                    : (n_width / 2 >= kStoreCols ? n_width / 2 : kStoreCols);
}
// fp32 partial sum of one epilogue warp (32 rows x its column group) and of
// a whole CTA (all its active epilogue warps) for a full-width tile.
__host__ __device__ constexpr uint32_t epi_warp_partial_bytes(int bn, int groups) {
  return 32u * static_cast<uint32_t>(epi_group_cols(bn, groups)) * 4u;
}
__host__ __device__ constexpr size_t epi_cta_partial_bytes(int bn, int groups) {
  return static_cast<size_t>(4 * (groups < 2 ? 1 : 2)) * epi_warp_partial_bytes(bn, groups);
}

// Shared memory a CTA needs for a given tile width / ring depth / staging
// (store_bufs buffers for each of the epi_groups x 4 active epilogue warps);
// with a CTA pair (cta_group 2) each CTA holds half of the tile's B rows.
// Dynamic shared memory of a kernel launch: `stages` K slices of A (a_rows
// rows: kBM, or 64 for a single row of single-CTA tiles with M <= 64) and B,
// the epilogue staging buffers and the barriers.
inline size_t kernel_smem_bytes(int bn, int stages, int store_bufs, int cta_group = 1,
                                int epi_groups = 1, int a_rows = kBM) {
  const size_t stage =
      static_cast<size_t>(a_rows) * kBK * 2 + static_cast<size_t>(bn / cta_group) * kBK * 2;
  return kAlignSlack + stage * static_cast<size_t>(stages) +
         static_cast<size_t>(4 * epi_groups) * store_bufs * kStoreBuf + kBarrierBytes;
}

}  // namespace spgemm
