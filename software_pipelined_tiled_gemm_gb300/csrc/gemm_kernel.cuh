// gemm_kernel.cuh -- persistent, warp-specialised sm_103a GEMM
//
//   C[M,N] = epi(A[M,K] . B^T), B stored N x K (or K x N), fp16/bf16 in,
//   fp32 accumulate in TMEM, fp16/bf16 (or fp32) out, epi in {none, tanh-GELU,
//   ReLU}.
//
// Structure (TileLang tutorial ch. 11 "pipelined_gemm.py", matmul_auto, for
// the tile loop; Mosaic GPU pipelining guide, "Warp Specialization", for the
// split into a memory thread and compute threads):
//
//   warp 0  (one lane)  TMA producer: for every unit of work and every ring
//                       slot's worth of K (one or two 64-wide slices), wait
//                       until slot s is empty, then copy the A rows and B
//                       rows of those slices into slot s with 128-byte
//                       swizzling; the copy engine counts the bytes onto
//                       full[s].
//   warp 1  (one lane)  MMA issuer: wait full[s], issue 4 tcgen05.mma per
//                       slice (K = 16 each) into the unit's TMEM accumulator,
//                       then tcgen05.commit -> empty[s].  The slot is
//                       released only when those MMAs have finished reading
//                       it (the hazard the guide's delay_release covers), and
//                       the issuer never waits on its own MMAs.  After the
//                       unit's last slot: commit -> tmem_full[acc].
//   warps 2-5 (or 2-9)  epilogue, one (or two) warps per TMEM lane quarter
//                       (warp w may read lanes 32*(w%4) ..), each taking the
//                       unit's columns (or one half of them): wait
//                       tmem_full[acc]; for
//                       stream-K owners, add the other walker's fp32 partial;
//                       then tcgen05.ld 32 rows x 64 columns per step, add
//                       the bias (if any), apply the epilogue function,
//                       round, write a swizzled staging tile and send it out
//                       with a TMA store (or row-wise stores when C's pitch
//                       is not 16-byte aligned); then arrive on
//                       tmem_empty[acc].
//
// With two TMEM accumulators the epilogue of one unit overlaps the main loop
// of the next.  CTA pairs (cluster of 2, tcgen05.mma.cta_group::2) compute
// 256-row tiles: each CTA copies its own 128 rows of A and half of B's rows,
// and the even CTA issues the MMAs for both.  The CTAs (or pairs) are
// persistent walkers over a grouped ("rasterised") tile order that keeps
// `raster_group` tile rows together, so concurrently running walkers share A
// and B rows in L2; with serpentine K, alternate waves walk K downwards so
// that each starts on the slices its predecessor read last.  The last,
// partial wave is shared out stream-K (or cut into narrow tiles); a problem
// of few tiles splits each in two K halves on the two CTAs of a cluster,
// whose partial moves through distributed shared memory.  Operands larger
// than L2 have each CTA's first ring prefetched into L2 while the previous
// kernel in the stream finishes.
//
// Every wait is bounded by a wall-clock limit; a wait that runs out records
// GEMM_ERR_TIMEOUT in the status word and its role stops, after which the CTA
// drains its in-flight copies and MMAs and frees its TMEM.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "byte_shift.cuh"
#include "epilogue_math.cuh"
#include "kernel_params.h"
#include "ptx.cuh"

namespace spgemm {

static __device__ __noinline__ void record_error(int* status, int code, int detail) {
  if (atomicCAS(status, 0, code) == 0) atomicExch(status + 1, detail);
}

// Range checks of the bounds-checked build (compiled with
// SPGEMM_BOUNDS_CHECKS=1).  SPGEMM_OUT_OF_BOUNDS(cond, p, what) is true when
// `cond` fails; it then records GEMM_ERR_BOUNDS and the check's identity
// `what` in the status word, the caller skips the access and ends its role,
// and the other roles' bounded waits run out -- no trap, the GPU stays
// usable.  In the normal build it is the constant false and `cond` is not
// evaluated.
__device__ __forceinline__ bool check_failed(const Params& p, int what) {
  record_error(p.status, kStatusBounds, what);
  return true;
}
#define SPGEMM_OUT_OF_BOUNDS(cond, p, what) \
  (SPGEMM_BOUNDS_CHECKS && !(cond) && ::spgemm::check_failed((p), (what)))

// Suspend-time hint of the long waits (an epilogue warp waits for most of a
// tile's main loop): wake on the phase, not on a short default limit.
constexpr uint32_t kLongWaitHintNs = 1000000u;

// Wait for the phase of parity `parity` of barrier `bar`; false on timeout.
// kLong: the wait is expected to be long (suspend-time hint).
template <bool kLong = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const Params& p,
                                             int detail) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!(kLong ? ptx::mbar_try_wait_sleep(bar, parity, kLongWaitHintNs)
                 : ptx::mbar_try_wait(bar, parity))) {
    if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
      record_error(p.status, kStatusTimeout, detail);
      return false;
    }
  }
  return true;
}

// As wait_bounded, with cluster-scope acquire when other CTAs arrive on `bar`.
template <int CG>
__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                     const Params& p, int detail) {
  if constexpr (CG == 1) {
    return wait_bounded(bar, parity, p, detail);
  } else {
    if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait_cluster(bar, parity)) {
      if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
        record_error(p.status, kStatusTimeout, detail);
        return false;
      }
    }
    return true;
  }
}

__device__ __forceinline__ int ld_acquire_gpu(const int* ptr) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

// Wait (bounded) until another walker has raised *flag after publishing its
// partial sum.
__device__ __forceinline__ bool wait_flag(const int* flag, const Params& p, int detail) {
  if (ld_acquire_gpu(flag) != 0) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (ld_acquire_gpu(flag) == 0) {
    __nanosleep(32);
    if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
      record_error(p.status, kStatusTimeout, detail);
      return false;
    }
  }
  return true;
}

// Grouped tile order: tiles are taken `raster_group` tile rows at a time,
// column by column inside a group.
__device__ __forceinline__ void tile_coords(int t, const Params& p, int& mb, int& nb) {
  const int per_group = p.raster_group * p.tiles_n;
  const int g = t / per_group;
  const int first_m = g * p.raster_group;
  const int rows = min(p.tiles_m - first_m, p.raster_group);
  const int r = t - g * per_group;
  mb = first_m + r % rows;
  nb = r / rows;
}

// One piece of work for a walker (a CTA, or a CTA pair).
struct Unit {
  int tile;    // raster index of the output tile
  int sub;     // narrow tail tile index along N, or -1 for a full-width tile
  int k0, k1;  // K slices [k0, k1) of this piece
  int role;    // kWhole, kContrib (partial sum for another walker), kOwner (adds it, stores)
  int seq;     // running count of this walker's units
  int wave;    // wave of whole tiles (walker's n-th whole tile), 0 for stream-K pieces
  int skt;     // stream-K tile index of a stream-K piece, -1 otherwise
};
constexpr int kWhole = 0, kContrib = 1, kOwner = 2;

// Enumerates a walker's units: its whole tiles (and narrow tail tiles),
// walker, walker + walkers, ...; and, with stream-K, its contiguous share
// [begin, end) of the sk_tiles * k_blocks K iterations of the stream-K
// tiles -- after the whole tiles, or before them with Params::sk_first.
struct UnitIter {
  int u;
  int walkers;
  int seq = 0;
  int64_t sk_it = 0, sk_end = 0;
  __device__ UnitIter(int walker, int walkers_, const Params& p) : u(walker), walkers(walkers_) {
    if (p.sk_tiles > 0) {
      const int64_t total = static_cast<int64_t>(p.sk_tiles) * p.k_blocks;
      sk_it = total * walker / walkers;
      sk_end = total * (walker + 1) / walkers;
    }
  }
  __device__ bool next(const Params& p, Unit& x) {
    if (p.sk_first && sk_it < sk_end) return next_sk(p, x);
    if (u < p.num_units) {
      x.wave = u / walkers;
      x.skt = -1;
      if (u < p.dp_tiles) {
        x.tile = p.sk_first ? p.sk_tiles + u : u;
        x.sub = -1;
      } else {
        const int v = u - p.dp_tiles;
        x.tile = p.dp_tiles + v / p.tail_splits;
        x.sub = v - (v / p.tail_splits) * p.tail_splits;
      }
      x.k0 = 0;
      x.k1 = p.k_blocks;
      x.role = kWhole;
      x.seq = seq++;
      u += walkers;
      return true;
    }
    if (sk_it < sk_end) return next_sk(p, x);
    return false;
  }
  // The next piece of this walker's stream-K share.
  __device__ bool next_sk(const Params& p, Unit& x) {
    const int64_t tl = sk_it / p.k_blocks;
    x.skt = static_cast<int>(tl);
    x.wave = 0;
    x.tile = p.sk_first ? static_cast<int>(tl) : p.dp_tiles + static_cast<int>(tl);
    x.sub = -1;
    x.k0 = static_cast<int>(sk_it - tl * p.k_blocks);
    const int64_t left = sk_end - sk_it;
    x.k1 = static_cast<int>(x.k0 + left < p.k_blocks ? x.k0 + left : p.k_blocks);
    x.role = (x.k0 == 0 && x.k1 == p.k_blocks) ? kWhole : (x.k0 > 0 ? kContrib : kOwner);
    x.seq = seq++;
    sk_it += x.k1 - x.k0;
    return true;
  }
};

// First K slice of a whole unit's loop: 0, or spread over the K range.
__device__ __forceinline__ int k_start(const Unit& x, int walker, int walkers, const Params& p) {
  if (!p.k_rotate || x.role != kWhole) return 0;
  const int n = walkers < p.num_units ? walkers : p.num_units;
  const int idx = (walker + x.seq * walkers) % n;
  return static_cast<int>((static_cast<int64_t>(idx) * p.k_blocks) / n);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
  if (bf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Bias of one column (0 at or beyond N), as fp32.  Lane l fetches the
// columns col0 + l and col0 + 32 + l of a 64-column chunk: two coalesced
// 64-byte loads per warp, issued one chunk ahead of their use.
__device__ __forceinline__ float load_bias(const Params& p, int col, bool bf16) {
  if (col >= p.N) return 0.0f;
  const unsigned short bits = __ldg(static_cast<const unsigned short*>(p.bias) + col);
  return bf16 ? __bfloat162float(__ushort_as_bfloat16(bits)) : __half2float(__ushort_as_half(bits));
}

// r[j] += the bias of column j of the 32 (lane j holds it in `b`): every row
// (lane) adds the same 32 values, handed round by warp shuffles.
__device__ __forceinline__ void add_bias32(uint32_t (&r)[32], float b) {
#pragma unroll
  for (int j = 0; j < 32; ++j)
    r[j] = __float_as_uint(__uint_as_float(r[j]) + __shfl_sync(0xffffffffu, b, j));
}

// Epilogue function EPI on 32 fp32 accumulator values held as raw words:
// 1 tanh-GELU, 2 ReLU (max(x, 0), with -0 and NaN giving +0).  Callers pick
// EPI once per 64-column chunk, so the unrolled loop holds no per-element
// branch (a per-element switch cost 11-12 % at 4096^3).
template <int EPI>
__device__ __forceinline__ void apply_epilogue32(uint32_t (&r)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    float x = __uint_as_float(r[j]);
    if constexpr (EPI == 1) x = gelu_tanh(x);
    if constexpr (EPI == 2) x = relu(x);
    r[j] = __float_as_uint(x);
  }
}

// Store one 32-row x 128-byte block of C held as 32 words per lane (lane =
// row, words = the row's 128 bytes): `esize`-byte elements starting at
// column col0 of rows row0 .. row0+31.  The block goes through the warp's
// staging buffer in the layout of a 128-byte-swizzled TMA box (16-byte chunk
// j of row r at j ^ (r % 8): bank-conflict free), then out with one TMA store
// (double-buffered staging), or -- when C's pitch or address is not 16-byte
// aligned -- by the warp's own stores.  A whole block of 16-bit elements
// goes four rows per step: eight lanes per row, lane j writing the row's
// 16-byte-aligned chunk j (realigned from two staging chunks), and one
// 2-byte store per lane for the row's unaligned head and tail, which
// together always hold 8 elements.  A block cut by the edge of C goes row by
// row, element by element.
__device__ __forceinline__ void store_rows(const uint32_t (&w)[32], const Params& p,
                                           const CUtensorMap& tmC, uint8_t* my_stage, int& buf,
                                           int lane, int row0, int col0, int esize) {
  if (p.tma_store) {
    // The staging buffer about to be written must have been read out by the
    // store issued store_bufs blocks ago.
    if (lane == 0) {
      if (p.store_bufs == 2)
        ptx::bulk_wait_group_read<1>();
      else
        ptx::bulk_wait_group_read<0>();
    }
    __syncwarp();
    uint8_t* sb = my_stage + buf * kStoreBuf;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t off = lane * 128u + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4);
      *reinterpret_cast<uint4*>(sb + off) = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      ptx::tma_store_2d(&tmC, ptx::smem_addr(sb), col0, row0);
      ptx::bulk_commit_group();
    }
    buf = (buf + 1 == p.store_bufs) ? 0 : buf + 1;
  } else {
    __syncwarp();  // the previous block's reads of the buffer are done
    uint8_t* sb = my_stage;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t off = lane * 128u + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4);
      *reinterpret_cast<uint4*>(sb + off) = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    }
    __syncwarp();
    const int per_row = 128 / esize;                       // elements in the block's row
    const int ncols = min(per_row, p.N - col0);
    const int nrows = min(32, p.M - row0);
    if (esize == 2 && ncols == 64 && nrows == 32) {
      const uint32_t j = static_cast<uint32_t>(lane) & 7u;  // the 16-byte chunk this lane writes
#pragma unroll 1
      for (int r4 = 0; r4 < 32; r4 += 4) {
        const uint32_t r = static_cast<uint32_t>(r4 + (lane >> 3));
        uint8_t* crow = reinterpret_cast<uint8_t*>(p.C) + (static_cast<int64_t>(row0 + r) * p.ldc + col0) * 2;
        const uint32_t a = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(crow) & 15u);  // even
        const uint8_t* srow = sb + r * 128u;
        const uint32_t sw = r & 7u;                          // the row's chunk swizzle
        if (a == 0) {
          // Aligned row: chunk j is staging chunk j.
          *reinterpret_cast<uint4*>(crow + 16u * j) = *reinterpret_cast<const uint4*>(srow + ((j ^ sw) << 4));
        } else {
          // Aligned chunk j (1..7) holds row bytes [16j - a, 16j - a + 16):
          // the end of staging chunk j - 1 and the start of chunk j.
          if (j != 0) {
            const uint4 lo = *reinterpret_cast<const uint4*>(srow + (((j - 1u) ^ sw) << 4));
            const uint4 hi = *reinterpret_cast<const uint4*>(srow + ((j ^ sw) << 4));
            *reinterpret_cast<uint4*>(crow - a + 16u * j) = shift_window(lo, hi, 16u - a);
          }
          // Head (row elements 0 .. h-1, h = (16 - a) / 2) and tail (the last
          // a / 2 elements): 8 elements, one per lane of the row.
          const uint32_t h = (16u - a) >> 1;
          const uint32_t e = j < h ? j : 64u - 8u + j;       // row element of this lane
          const uint32_t byte = 2u * e;
          *reinterpret_cast<uint16_t*>(crow + byte) =
              *reinterpret_cast<const uint16_t*>(srow + ((((byte >> 4) ^ sw)) << 4) + (byte & 15u));
        }
      }
      return;
    }
#pragma unroll 1
    for (int r = 0; r < nrows; ++r) {
      uint8_t* crow = reinterpret_cast<uint8_t*>(p.C) +
                      (static_cast<int64_t>(row0 + r) * p.ldc + col0) * esize;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int cc = lane + 32 * h;                      // element index in the row
        if (cc < ncols) {
          const uint32_t byte = static_cast<uint32_t>(cc * esize);
          const uint32_t off = static_cast<uint32_t>(r) * 128u +
                               (((byte >> 4) ^ (static_cast<uint32_t>(r) & 7u)) << 4) + (byte & 15u);
          if (esize == 2)
            *reinterpret_cast<uint16_t*>(crow + cc * 2) = *reinterpret_cast<const uint16_t*>(sb + off);
          else
            *reinterpret_cast<uint32_t*>(crow + cc * 4) = *reinterpret_cast<const uint32_t*>(sb + off);
        }
      }
    }
  }
}

// BN: output tile width.  CG: CTAs per tile (1, or 2 for a CTA pair that
// computes a 256 x BN tile with cta_group::2 MMAs: each CTA loads its own 128
// rows of A and BN/2 rows of B, the even CTA issues the MMAs for both, and
// each CTA's TMEM receives its own 128 rows of the accumulator).
// kSplit: this instance can run narrow tail tiles (BN / tail_splits wide,
// B loaded through tmBt) and stream-K pieces; the instance used by plans
// that need neither has that code compiled out.
// kKN: B is stored K x N and read MN-major (see Params::b_kn).
// kStream: every element of B is read once, and B's copies carry an
// evict-first L2 policy (see Params::b_stream).
// kSub: 64-wide K slices per ring slot.  With 2, one full/empty barrier
// round trip covers 8 MMAs instead of 4 (the slot holds two slices of A and
// two of B side by side); p.stages and p.k_blocks count slots.
// kEpiG: epilogue column groups, 1 (warps 2-5, 192 threads) or 2 (warps 2-9,
// 320 threads: two warps per TMEM lane quarter, each taking half of a unit's
// columns).  Eight warps halve an exposed epilogue; where the epilogue hides
// behind a long main loop, four run faster (a second epilogue warp on the
// MMA issuer's sub-partition costs ~0.5-1 % of the cycles at 8192^3).
template <int BN, int CG, bool kSplit, bool kKN, bool kStream, int kSub, int kEpiG>
__global__ void __launch_bounds__(kernel_threads(kEpiG), 1)
    gemm_tn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmBt, const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmBp, const Params p) {
  static_assert(CG == 1 || CG == 2, "CTA group of 1 or 2");
  static_assert(kSub == 1 || kSub == 2, "one or two K slices per slot");
  constexpr int kBRows = BN / CG;                    // B rows this CTA loads
  constexpr uint32_t kStageB = kBRows * kBK * 2;     // B bytes of one K slice
  constexpr uint32_t kBBlocks = kBRows / 64;           // 64-column blocks of a K x N B slice
  // A bytes of one K slice in the ring: the whole 128-row box, except that a
  // single row of single-CTA tiles with M <= 64 copies (and keeps) only 64
  // rows -- the MMA's rows 64-127 then read the next bytes of the slot, and
  // feed only output rows >= M, which are never stored.  The freed space
  // holds more slices (M = 64: 8 slices of 128-column B instead of 6).
  const uint32_t slice_a = kStream ? static_cast<uint32_t>(p.a_box_rows) * (kBK * 2u) : kStageA;
  const uint32_t slot_a = slice_a * kSub;              // A part of a slot
  const uint32_t slot_bytes = slot_a + kStageB * kSub;  // bytes per slot, this CTA
  constexpr int kTileM = kBM * CG;                   // output rows per tile
  static_assert(kEpiG == 1 || kEpiG == 2, "one or two epilogue column groups");
  constexpr int epi_groups = kEpiG;  // epilogue column groups (4 x kEpiG epilogue warps)
  // fp32 partial of one epilogue warp (32 rows x its column group)
  const uint32_t warp_partial = epi_warp_partial_bytes(BN, epi_groups);

  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment: the 128-byte swizzle pattern repeats every 1024 B
  // and the MMA descriptors assume atoms start on that boundary.
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_addr(smem);

  const int S = p.stages;
  const uint32_t ring_bytes = static_cast<uint32_t>(S) * slot_bytes;
  uint8_t* staging = smem + ring_bytes;
  const uint32_t staging_bytes = 4u * epi_groups * p.store_bufs * kStoreBuf;
  const uint32_t bar_base = sbase + ring_bytes + staging_bytes;
  // Ring, staging, barriers and the TMEM address slot inside the launch's
  // dynamic shared memory (every thread of every CTA decides alike, so all
  // leave before any barrier, TMEM allocation or cluster synchronisation).
  if (SPGEMM_OUT_OF_BOUNDS(S >= 1 && S <= kMaxStages && p.store_bufs >= 1 && p.store_bufs <= 2 &&
                               (sbase - raw_addr) + ring_bytes + staging_bytes +
                                       8u * (2 * kMaxStages + 5 + 2 * kEpiWarps) + 4u <=
                                   ptx::dynamic_smem_bytes(),
                           p, kCheckSmemLayout))
    return;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (kMaxStages + s); };
  auto tfull_bar = [&](int a) { return bar_base + 8u * (2 * kMaxStages + a); };
  auto tempty_bar = [&](int a) { return bar_base + 8u * (2 * kMaxStages + 2 + a); };
  const uint32_t done_bar = bar_base + 8u * (2 * kMaxStages + 4);
  auto fix_bar = [&](int e) { return bar_base + 8u * (2 * kMaxStages + 5 + e); };
  // Cluster split: the owner tells the contributor its ring is free.
  auto free_bar = [&](int e) { return bar_base + 8u * (2 * kMaxStages + 5 + kEpiWarps + e); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + ring_bytes + staging_bytes +
                                                    8u * (2 * kMaxStages + 5 + 2 * kEpiWarps));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t tmem_cols = static_cast<uint32_t>(p.tmem_cols);
  // Position in the CTA pair (always 0 without one).
  const uint32_t rank = (CG == 2) ? ptx::cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int walker = static_cast<int>(blockIdx.x) / CG;
  const int walkers = static_cast<int>(gridDim.x) / CG;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull_bar(a), 1);
      // Every epilogue warp of every CTA of the tile releases the accumulator.
      ptx::mbar_init(tempty_bar(a), 4 * kEpiG * CG);
    }
    ptx::mbar_init(done_bar, 1);
    for (int q = 0; q < kEpiWarps; ++q) {
      ptx::mbar_init(fix_bar(q), 1);
      ptx::mbar_init(free_bar(q), 1);
    }
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
    if (kSplit) ptx::tma_prefetch_desc(&tmBt);
    if (p.tma_store) ptx::tma_prefetch_desc(&tmC);
  }
  // Warm L2 with the slices the ring will hold first (operands that do not
  // stay in L2, see Params::l2_prefetch_first).  The first epilogue warp,
  // idle until the first accumulator is full, issues it before its wait on
  // the previous kernel: it only moves lines into L2, the device's point of
  // coherence (a line the previous kernel still writes is updated there),
  // and the ring's own copies are issued after the producer's wait.  Issued
  // by thread 0 before the CTA-wide set-up barrier instead, it delayed the
  // other roles' start: skinny 64 x 8192 x 8192 back to back 26.35 -> 25.60
  // us with it here (8192^3, the GELU layer and the ragged shape 0.2-0.4 %
  // faster too).
  auto prefetch_first_ring = [&]() {
    UnitIter it0(walker, walkers, p);
    Unit x0;
    if (!it0.next(p, x0)) return;
    int mb, nb;
    tile_coords(x0.tile, p, mb, nb);
    const bool narrow = kSplit && x0.sub >= 0;
    const int n_width = narrow ? BN / p.tail_splits : BN;
    const int a_row = mb * kTileM + static_cast<int>(rank) * kBM;
    const int b_row = nb * BN + (narrow ? x0.sub * n_width : 0) + static_cast<int>(rank) * (n_width / CG);
    const void* tmb = narrow ? static_cast<const void*>(&tmBt) : static_cast<const void*>(&tmB);
    const int nk = x0.k1 - x0.k0;
    const int kr = k_start(x0, walker, walkers, p);
    for (int i = 0; i < S && i < nk; ++i) {
      const int kb = x0.k0 + (kr + i) % nk;
#pragma unroll
      for (int sub = 0; sub < kSub; ++sub) {
        const int kx = (kb * kSub + sub) * kBK;
        ptx::tma_prefetch_l2_2d(&tmA, kx, a_row);
        if constexpr (!kKN)
          ptx::tma_prefetch_l2_2d(tmb, kx, b_row);
        else
          ptx::tma_prefetch_l2_4d(tmb, 0, 0, b_row / 64, kx / 8);
      }
    }
  };
  if (warp == 1) {
    ptx::tmem_alloc<CG>(ptx::smem_addr(tmem_slot), tmem_cols);
    ptx::tmem_relinquish<CG>();
  }
  ptx::tc_fence_before_sync();
  // Peer barriers must be initialised before any remote arrive / TMA.
  if (CG == 2 || (kSplit && p.sk_cluster))
    ptx::cluster_sync();
  else
    __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  // Programmatic dependent launch: the set-up above touched no global memory
  // and may overlap the previous kernel's tail.  Each role waits for that
  // kernel to finish right before its own first global-memory access: the
  // producer before its first copy (so the work of finding its first unit
  // overlaps the previous kernel too), the epilogue warps before anything
  // else.  The MMA issuer reads only shared and tensor memory and does not
  // wait.
  ptx::pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;  // per-slot: used at all / parity of last use
      // B read once (a single row of tiles): evict its lines from L2 first.
      const uint64_t pol_b = kStream ? ptx::l2_policy_evict_first() : 0;
      bool ok = true;
      bool waited = false;  // on the previous kernel in the stream
      UnitIter it(walker, walkers, p);
      Unit x;
      while (ok && it.next(p, x)) {
        int mb, nb;
        tile_coords(x.tile, p, mb, nb);
        if (SPGEMM_OUT_OF_BOUNDS(x.tile >= 0 && x.tile < p.num_tiles && mb >= 0 && mb < p.tiles_m &&
                                     nb >= 0 && nb < p.tiles_n,
                                 p, kCheckTile) ||
            SPGEMM_OUT_OF_BOUNDS(x.k0 >= 0 && x.k0 < x.k1 && x.k1 <= p.k_blocks, p, kCheckKSlice)) {
          ok = false;
          break;
        }
        const bool narrow = kSplit && x.sub >= 0;
        const int n_width = narrow ? BN / p.tail_splits : BN;   // columns of this unit
        const int b_rows = n_width / CG;                        // B rows this CTA loads
        const int a_row = mb * kTileM + static_cast<int>(rank) * kBM;
        const int b_row = nb * BN + (narrow ? x.sub * n_width : 0) + static_cast<int>(rank) * b_rows;
        const void* tmb = narrow ? static_cast<const void*>(&tmBt) : static_cast<const void*>(&tmB);
        const uint32_t bytes =
            (static_cast<uint32_t>(p.a_box_rows) * kBK * 2u + static_cast<uint32_t>(b_rows) * kBK * 2u) *
            CG * kSub;
        const int nk = x.k1 - x.k0;
        const int kr = k_start(x, walker, walkers, p);
        const bool down =
            p.k_serpentine && ((p.sk_first ? x.wave : x.seq) & 1) && x.role == kWhole;
        for (int i = 0, kf = x.k0 + kr; i < nk; ++i, kf = (kf + 1 == x.k1) ? x.k0 : kf + 1) {
          const int kb = down ? x.k1 - 1 - i : kf;  // K slot this iteration copies
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, p, kDetailProducerEmpty)) {
            ok = false;
            break;
          }
          if (kSub == 1 && p.prefetch_kb > 0 && ((kb - x.k0) & (kPrefetchSlices - 1)) == 0) {
            // L2 prefetch of this unit's B rows, prefetch_kb slices ahead (wrapping
            // with the rotated K loop), 4 slices per request.
            int pk = kb + p.prefetch_kb;
            if (pk >= x.k1) pk -= (x.k1 - x.k0);
            if (pk >= x.k0 && pk < x.k1) ptx::tma_prefetch_l2_2d(&tmBp, pk * kBK, b_row);
          }
          const uint32_t sa = sbase + stage * slot_bytes;
          // Copy coordinates: the K slot inside the unit's range, the first K
          // element 16-byte aligned (x of a tiled copy) and inside the K
          // extent, the rows inside the tile grid.  Test hook 2 makes this
          // check fail for CTA 0's first copy (its coordinates are valid).
          {
            const int kx_first = kb * kSub * kBK, kx_last = (kb * kSub + kSub - 1) * kBK;
            const bool forced = p.inject_fault == 2 && blockIdx.x == 0 && x.seq == 0 && i == 0;
            if (SPGEMM_OUT_OF_BOUNDS(kb >= x.k0 && kb < x.k1 && stage < S, p, kCheckKSlice) ||
                SPGEMM_OUT_OF_BOUNDS(!forced && kx_first >= 0 && (kx_first & 7) == 0 &&
                                         kx_last < p.k_blocks * kSub * kBK && a_row >= 0 &&
                                         a_row < p.tiles_m * kTileM && b_row >= 0 &&
                                         b_row < p.tiles_n * BN && (!kKN || (b_row & 63) == 0),
                                     p, kCheckTmaCoord)) {
              ok = false;
              break;
            }
          }
          if (!waited) {
            ptx::pdl_wait_prior_grid();
            waited = true;
          }
          // Test hook: the first slice of CTA 0 is announced but never copied.
          const bool skip = p.inject_fault == 1 && blockIdx.x == 0 && x.seq == 0 && i == 0;
          if constexpr (CG == 2) {
            // Both CTAs' copies count on the leader's full barrier; only the
            // leader announces the bytes (of both CTAs).
            const uint32_t fb = ptx::map_shared_rank(full_bar(stage), 0);
            if (leader) ptx::mbar_arrive_expect_tx(full_bar(stage), bytes);
            static_assert(!kStream, "streamed B is a single-CTA instance");
#pragma unroll
            for (int sub = 0; sub < kSub; ++sub) {
              if (skip) break;
              const int kx = (kb * kSub + sub) * kBK;  // first K element of this slice
              const uint32_t da = sa + sub * slice_a, db = sa + slot_a + sub * kStageB;
              ptx::tma_load_2d_pair(da, &tmA, kx, a_row, fb);
              if constexpr (!kKN)
                ptx::tma_load_2d_pair(db, tmb, kx, b_row, fb);
              else  // (64 columns, 8 K rows, column blocks, K groups of 8)
                ptx::tma_load_4d_pair(db, tmb, 0, 0, b_row / 64, kx / 8, fb);
            }
          } else {
            ptx::mbar_arrive_expect_tx(full_bar(stage), bytes);
#pragma unroll
            for (int sub = 0; sub < kSub; ++sub) {
              if (skip) break;
              const int kx = (kb * kSub + sub) * kBK;
              const uint32_t da = sa + sub * slice_a, db = sa + slot_a + sub * kStageB;
              ptx::tma_load_2d(da, &tmA, kx, a_row, full_bar(stage));
              if constexpr (!kKN && !kStream)
                ptx::tma_load_2d(db, tmb, kx, b_row, full_bar(stage));
              else if constexpr (!kKN)
                ptx::tma_load_2d_hint(db, tmb, kx, b_row, full_bar(stage), pol_b);
              else if constexpr (!kStream)
                ptx::tma_load_4d(db, tmb, 0, 0, b_row / 64, kx / 8, full_bar(stage));
              else
                ptx::tma_load_4d_hint(db, tmb, 0, 0, b_row / 64, kx / 8, full_bar(stage), pol_b);
            }
          }
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every copy this CTA pair started must have landed before it exits: the
      // leader's full barriers count the bytes of both CTAs (the final
      // cluster barrier keeps the peer resident until then).
      if (leader) {
        for (int s = 0; s < S; ++s)
          if (issued & (1u << s))
            wait_bounded(full_bar(s), (issued_parity >> s) & 1u, p, kDetailProducerDrain);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      UnitIter it(walker, walkers, p);
      Unit x;
      while (ok && it.next(p, x)) {
        const uint32_t idesc = (kSplit && x.sub >= 0) ? p.idesc_tail : p.idesc;
        if (!wait_bounded_cluster<CG>(tempty_bar(acc), acc_phase ^ 1u, p, kDetailMmaAccEmpty))
          break;
        ptx::tc_fence_after_sync();
        if (SPGEMM_OUT_OF_BOUNDS(acc >= 0 && acc < p.num_acc && (acc + 1) * BN <= p.tmem_cols, p,
                                 kCheckMmaTmem))
          break;
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        const int nk = x.k1 - x.k0;
        for (int kb = 0; kb < nk; ++kb) {  // iteration count (slices may be rotated)
          if (!wait_bounded(full_bar(stage), phase, p, kDetailMmaFull) ||
              SPGEMM_OUT_OF_BOUNDS(stage >= 0 && stage < S, p, kCheckMmaSlot)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after_sync();
          const uint32_t sa = sbase + stage * slot_bytes;
          const uint64_t a_desc = ptx::smem_desc_k_sw128(sa);
          // K-major B: +32 B per 16-wide K step inside the swizzled row (+2 in
          // 16-byte units).  MN-major B (atoms [K group][column block], the
          // column blocks of one K group adjacent): +2 K groups per step.
          const uint64_t b_desc =
              kKN ? ptx::smem_desc_mn_sw128(sa + slot_a, 1024u, kBBlocks * 1024u)
                  : ptx::smem_desc_k_sw128(sa + slot_a);
          constexpr uint32_t b_step = kKN ? 2u * kBBlocks * 1024u / 16u : 2u;
#pragma unroll
          for (int k = 0; k < kSub * (kBK / kUmmaK); ++k) {
            // Within a slice, +32 bytes along K inside the 128-byte swizzled
            // row = +2 in the descriptor's address field (16-byte units); the
            // second slice of a slot starts slice_a (A) / kStageB (B) later.
            // K x N B: the slices' row groups follow each other, +2 groups
            // per step throughout.
            const uint32_t sub = static_cast<uint32_t>(k) / 4u, kk = static_cast<uint32_t>(k) % 4u;
            const uint64_t ad = a_desc + sub * (slice_a / 16u) + 2u * kk;
            const uint64_t bd = kKN ? b_desc + b_step * static_cast<uint32_t>(k)
                                    : b_desc + sub * (kStageB / 16u) + 2u * kk;
            ptx::mma_f16_ss<CG>(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          if constexpr (CG == 2)
            ptx::mma_commit_multicast_pair(empty_bar(stage), 0x3);
          else
            ptx::mma_commit<1>(empty_bar(stage));
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (CG == 2)
          ptx::mma_commit_multicast_pair(tfull_bar(acc), 0x3);
        else
          ptx::mma_commit<1>(tfull_bar(acc));
        if (++acc == p.num_acc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // All MMAs this thread issued must be complete before TMEM is freed.
      ptx::mma_commit<CG>(done_bar);
      wait_bounded(done_bar, 0, p, kDetailMmaDrain);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- epilogue --
    // Warp 2 + e: TMEM lane quarter q (rows q*32 .. q*32+31 of the CTA's
    // accumulator) and column group g = e / 4 of every unit.  Stream-K
    // partials, flags and fix-up barriers are per warp e.
    if (warp == 2 && lane == 0 && p.l2_prefetch_first) prefetch_first_ring();
    ptx::pdl_wait_prior_grid();  // bias, workspace, flags and C are global
    const int q = warp & 3;       // TMEM lane quarter this warp may access
    const int ew = warp - 2;      // epilogue warp index: staging, partials, flags
    const int g = ew / 4;         // column group
    uint8_t* my_stage = staging + ew * p.store_bufs * kStoreBuf;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t fix_phase = 0;
    int buf = 0;
    const bool bf16 = p.bf16 != 0;
    UnitIter it(walker, walkers, p);
    Unit x;
    while (it.next(p, x)) {
      int mb, nb;
      tile_coords(x.tile, p, mb, nb);
      const bool narrow = kSplit && x.sub >= 0;
      const int n_width = narrow ? BN / p.tail_splits : BN;
      const int n0 = nb * BN + (narrow ? x.sub * n_width : 0);
      // This warp's columns [c_lo, c_hi) of the unit (empty for a group not
      // in use and for the second group of a 64-wide unit); a full-width
      // unit gives every active warp warp_partial bytes of partial sum.
      const int gcols = epi_group_cols(n_width, epi_groups);
      const int c_lo = g * gcols;
      const int c_hi = c_lo + gcols < n_width ? c_lo + gcols : n_width;
      const bool has_cols = g < epi_groups && c_lo < c_hi;
      // Bias of the warp's first 64-column chunk, fetched before the
      // accumulator wait so its latency hides there (later chunks: one chunk
      // ahead).
      float nb0 = 0.0f, nb1 = 0.0f;
      if (p.bias != nullptr && x.role != kContrib && has_cols) {
        nb0 = load_bias(p, n0 + c_lo + lane, bf16);
        nb1 = load_bias(p, n0 + c_lo + 32 + lane, bf16);
      }
      int ready = 1;
      if (lane == 0) ready = wait_bounded<true>(tfull_bar(acc), acc_phase, p, kDetailEpiFull) ? 1 : 0;
      ready = __shfl_sync(0xffffffffu, ready, 0);
      if (!ready) break;
      ptx::tc_fence_after_sync();

      const int row0 = mb * kTileM + static_cast<int>(rank) * kBM + q * 32;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * BN);
      // Stream-K: this warp's fp32 partial of a shared tile, laid out
      // [column - c_lo][lane] (one coalesced 128-byte line per column).
      const uint32_t flag_idx =
          (static_cast<uint32_t>(x.skt) * CG + rank) * (4u * epi_groups) + ew;
      float* partial = (kSplit && x.role != kWhole)
                           ? p.sk_ws + static_cast<size_t>(flag_idx) * (warp_partial / 4u)
                           : nullptr;
      // TMEM columns, staging buffers, the C block, and (stream-K) the
      // partial's workspace slot and its shared-memory region.
      if (SPGEMM_OUT_OF_BOUNDS(acc >= 0 && acc < p.num_acc && c_hi <= BN &&
                                   (acc + 1) * BN <= p.tmem_cols,
                               p, kCheckEpiTmem) ||
          SPGEMM_OUT_OF_BOUNDS((ew + 1) * p.store_bufs * kStoreBuf <= staging_bytes, p,
                               kCheckStaging) ||
          SPGEMM_OUT_OF_BOUNDS(row0 >= 0 && row0 < p.tiles_m * kTileM && n0 >= 0 && (n0 & 63) == 0,
                               p, kCheckStore) ||
          SPGEMM_OUT_OF_BOUNDS(!kSplit || x.role == kWhole || p.sk_cluster ||
                                   (static_cast<int>(flag_idx) < p.sk_slots && p.sk_ws != nullptr),
                               p, kCheckPartial) ||
          SPGEMM_OUT_OF_BOUNDS(!kSplit || x.role == kWhole || (ew + 1) * warp_partial <= ring_bytes,
                               p, kCheckFixup))
        break;
      bool have_partial = false;
      if (kSplit && x.role == kContrib && p.sk_cluster) {
        // Cluster split: stage this warp's partial in this CTA's own idle
        // ring ([column][lane], the layout the owner reads), then, once the
        // owner's ring is free, bulk-copy it there; the bytes complete the
        // owner's fix-up barrier.  Rows >= M are never stored, so their warps
        // exchange nothing.  The final cluster barrier keeps this CTA (the
        // copy's source) alive until the owner has received the bytes.
        if (row0 < p.M && has_cols) {
          float* stage_out = reinterpret_cast<float*>(smem + ew * warp_partial);
#pragma unroll 1
          for (int c = c_lo; c < c_hi; c += 32) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(t_row + c, v);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j)
              stage_out[(c - c_lo + j) * 32 + lane] = __uint_as_float(v[j]);
          }
          ptx::fence_proxy_async_smem();  // generic writes -> the copy engine
          __syncwarp();
          int ok = 1;
          if (lane == 0) {
            // A walker holds one unit in this mode, so the barrier's first phase.
            ok = wait_bounded_cluster<2>(free_bar(ew), 0, p, kDetailSkFree) ? 1 : 0;
            if (ok)
              ptx::bulk_copy_to_peer(ptx::map_shared_rank(sbase + ew * warp_partial, 0),
                                     sbase + ew * warp_partial, warp_partial,
                                     ptx::map_shared_rank(fix_bar(ew), 0));
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
        }
      } else if (kSplit && x.role == kContrib) {
        // Publish the partial sum of K slices [k0, k1) and raise the flag.
        if (has_cols) {
#pragma unroll 1
          for (int c = c_lo; c < c_hi; c += 32) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(t_row + c, v);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j)
              __stcg(partial + (c - c_lo + j) * 32 + lane, __uint_as_float(v[j]));
          }
          __threadfence();
          __syncwarp();
          if (lane == 0) atomicAdd(p.sk_flags + flag_idx, 1);
        }
      } else if (kSplit && x.role == kOwner && p.sk_cluster) {
        // Cluster split: this walker's MMAs are done (accumulator full), so
        // its ring is idle; let the contributor copy its partial there.
        if (row0 < p.M && has_cols) {
          int ok = 1;
          if (lane == 0) {
            // Arm the fix-up barrier for the partial's bytes before telling
            // the contributor that the ring may be written.
            ptx::mbar_arrive_expect_tx(fix_bar(ew), warp_partial);
            ptx::mbar_arrive_cluster(ptx::map_shared_rank(free_bar(ew), 1));
            ok = wait_bounded_cluster<2>(fix_bar(ew), fix_phase, p, kDetailSkCopy) ? 1 : 0;
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          // Every lane acquires the contributor's writes (the phase is complete).
          (void)ptx::mbar_try_wait_cluster(fix_bar(ew), fix_phase);
          fix_phase ^= 1u;
          have_partial = true;
        }
      } else if (kSplit && x.role == kOwner && has_cols && p.sk_first) {
        // The other walker's partial was its first piece, long published:
        // wait for its flag (usually already raised) and read the partial
        // from L2 in the adds below; the ring is busy with the next tile.
        int ok = 1;
        if (lane == 0) ok = wait_flag(p.sk_flags + flag_idx, p, kDetailSkFlag) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        (void)ld_acquire_gpu(p.sk_flags + flag_idx);  // every lane acquires the partial
        have_partial = true;
      } else if (kSplit && x.role == kOwner && has_cols) {
        // The other walker's partial (K slices [k1, k_blocks)) was written at
        // the start of its range.  This is the last unit of this walker, so
        // the ring is idle: bulk-copy the partial into it.
        int ok = 1;
        if (lane == 0) {
          ok = wait_flag(p.sk_flags + flag_idx, p, kDetailSkFlag) ? 1 : 0;
          if (ok) {
            p.sk_flags[flag_idx] = 0;  // ready for the next launch
            ptx::mbar_arrive_expect_tx(fix_bar(ew), warp_partial);
            ptx::bulk_load(sbase + ew * warp_partial, partial, warp_partial, fix_bar(ew));
            ok = wait_bounded(fix_bar(ew), fix_phase, p, kDetailSkCopy) ? 1 : 0;
          }
        }
        fix_phase ^= 1u;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        have_partial = ok != 0;
        if (!have_partial) break;
      }
      if ((!kSplit || x.role != kContrib) && row0 < p.M && has_cols) {
        const float* fix = reinterpret_cast<const float*>(smem + ew * warp_partial);
#pragma unroll 1
        for (int cc = c_lo; cc < c_hi; cc += kStoreCols) {  // 64-column chunks
          const int col0 = n0 + cc;
          if (col0 >= p.N) break;
          const float b0 = nb0, b1 = nb1;
          if (p.bias != nullptr && cc + kStoreCols < c_hi) {
            nb0 = load_bias(p, col0 + kStoreCols + lane, bf16);
            nb1 = load_bias(p, col0 + kStoreCols + 32 + lane, bf16);
          }
          uint32_t r0[32], r1[32];
          ptx::tmem_ld_32x32b_x32(t_row + cc, r0);
          ptx::tmem_ld_32x32b_x32(t_row + cc + 32, r1);
          ptx::tmem_wait_ld();
          if (kSplit && have_partial && p.sk_first && !p.sk_cluster) {
            // own slices first, then the partial (from L2): a fixed order on every run
            const int cb = cc - c_lo;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              r0[j] = __float_as_uint(__uint_as_float(r0[j]) + __ldcg(partial + (cb + j) * 32 + lane));
              r1[j] = __float_as_uint(__uint_as_float(r1[j]) +
                                      __ldcg(partial + (cb + 32 + j) * 32 + lane));
            }
          } else if (kSplit && have_partial) {
            // own slices first, then the partial: a fixed order on every run
            const int cb = cc - c_lo;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              r0[j] = __float_as_uint(__uint_as_float(r0[j]) + fix[(cb + j) * 32 + lane]);
              r1[j] = __float_as_uint(__uint_as_float(r1[j]) + fix[(cb + 32 + j) * 32 + lane]);
            }
          }
          if (p.bias != nullptr) {  // after the partial: a fixed order on every run
            add_bias32(r0, b0);
            add_bias32(r1, b1);
          }
          // Epilogue function on the fp32 accumulator values.
          if (p.epilogue == 1) {
            apply_epilogue32<1>(r0);
            apply_epilogue32<1>(r1);
          } else if (p.epilogue == 2) {
            apply_epilogue32<2>(r0);
            apply_epilogue32<2>(r1);
          }
          const int halves = p.out_f32 ? 2 : 1;
#pragma unroll 1
          for (int h = 0; h < halves; ++h) {
            uint32_t pk[32];
            if (!p.out_f32) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                pk[j] = pack2(__uint_as_float(r0[2 * j]), __uint_as_float(r0[2 * j + 1]), bf16);
                pk[16 + j] = pack2(__uint_as_float(r1[2 * j]), __uint_as_float(r1[2 * j + 1]), bf16);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) pk[j] = h ? r1[j] : r0[j];
            }
            store_rows(pk, p, tmC, my_stage, buf, lane, row0, col0 + 32 * h, p.out_f32 ? 4 : 2);
          }
        }
      }
      if (kSplit && p.sk_first && !p.sk_cluster && x.role == kOwner && has_cols) {
        __syncwarp();                               // every lane has read the partial
        if (lane == 0) p.sk_flags[flag_idx] = 0;    // ready for the next launch
      }
      // This warp's TMEM reads of accumulator `acc` are complete (wait::ld).
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 2)
          ptx::mbar_arrive_cluster(ptx::map_shared_rank(tempty_bar(acc), 0));
        else
          ptx::mbar_arrive(tempty_bar(acc));
      }
      if (++acc == p.num_acc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) ptx::bulk_wait_group_all();
    __syncwarp();
  }

  ptx::tc_fence_before_sync();
  // Neither CTA of a cluster leaves while its peer may still touch its memory.
  if (CG == 2 || (kSplit && p.sk_cluster))
    ptx::cluster_sync();
  else
    __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc<CG>(tmem_base, tmem_cols);
  }
}

}  // namespace spgemm
