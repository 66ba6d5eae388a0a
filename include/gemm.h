/*
 * gemm.h -- C ABI of the GB300 (sm_103a) software-pipelined tiled GEMM.
 *
 *   C[i,j] = epi( sum_k A[i,k] * B[j,k] ),   0 <= i < M, 0 <= j < N
 *
 * Operation.  TileLang tutorial, chapter 11 ("Pipelining and autotuning"),
 * pipelined_gemm.py, kernel matmul_auto: A is an (M, K) tensor, B an (N, K)
 * tensor, C an (M, N) tensor; every (block_M, block_N) output tile clears a
 * float32 accumulator, walks the K dimension in block_K slices through a
 * num_stages-deep pipeline and multiplies with T.gemm(..., transpose_B=True);
 * the float32 tile is then written out in the 16-bit input type.  The inputs
 * are fp16 or bf16, the products are accumulated in fp32, and each output is
 * rounded once, to nearest even, to the input type.
 *
 * Epilogue.  GEMM_EPI_GELU_TANH applies the tanh-approximate GELU
 * 0.5 x (1 + tanh(0.7978845608 (x + 0.044715 x^3))) to the fp32 accumulator
 * before the rounding (the form written in the Triton lecture notes' "GeLU"
 * example and in the XLA:GPU emitters page's loop-emitter @gelu function).
 *
 * Pipelining.  `stages` is the depth of the shared-memory ring that the K
 * loop streams through -- num_stages in the TileLang tutorial,
 * max_concurrent_steps in the Mosaic GPU pipelining guide ("Pipelining with
 * Mosaic GPU").  A ring slot is handed back to the copy engine only when the
 * tensor-core instructions that read it have completed; this is the hazard
 * the guide's delay_release option exists for (refilling a slot that an
 * asynchronous matrix multiply has not finished reading).  GEMM_SINGLE_BUFFER is the tutorial's
 * matmul_plain contrast: one slot, one accumulator, so copies and math of
 * consecutive K slices cannot overlap.
 *
 * Layout.  All matrices are row-major and dense: A has K elements per row
 * (lda = K), B has K elements per row (ldb = K), C has N elements per row
 * (ldc = N).  Both operands are therefore K-contiguous ("K-major").  With
 * gemm_tuning_t.b_kn = 1, B is instead K x N (ldb = N) and the GEMM is
 * C = epi(A . B).
 * Element type of A and B is `dtype`; C has the same type, or fp32 when the
 * plan was created with gemm_tuning_t.out_f32 = 1.  Pointers A, B, C are device
 * pointers (cudaMalloc / torch CUDA tensors) on the plan's device, except for
 * gemm_run_host, which takes host pointers.
 *
 * Partial tiles.  Any M, N >= 0 and K >= 0 is accepted.  Out-of-range rows
 * and K columns contribute zero and out-of-range outputs are never written
 * (the masked loads and stores of the Triton lecture notes' matmul example).
 * When a row pitch or a base address is not 16-byte aligned, A and B are
 * first copied into plan-owned, padded device scratch and C is written with
 * plain masked stores instead of bulk tensor stores.
 *
 * Ownership.  The caller owns A, B, C and the stream.  A plan owns its
 * device status word, its padding scratch and (after the first
 * gemm_run_host) its device staging buffers; gemm_plan_destroy frees them.
 *
 * Threading.  A plan may be used from one host thread at a time and must not
 * have launches in flight on two streams at once.  Different plans are
 * independent.
 *
 * Errors.  Every entry point returns a gemm_status_t and never throws.
 * Argument errors are detected on the host before anything is launched.
 * Faults detected on the device (a pipeline wait that ran out its time
 * limit) are recorded in the plan's status word and reported by
 * gemm_plan_check.  gemm_run is asynchronous: a GEMM_OK return means the
 * work was enqueued.
 */
#ifndef SPGEMM_GEMM_H_
#define SPGEMM_GEMM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GEMM_OK = 0,
  GEMM_ERR_INVALID_ARG = 1,   /* null/negative/out-of-range argument, aliasing C with A or B */
  GEMM_ERR_UNSUPPORTED = 2,   /* device is not sm_103 / feature not built */
  GEMM_ERR_SMEM_BUDGET = 3,   /* requested stages/tile do not fit the shared-memory budget */
  GEMM_ERR_PLAN_MISMATCH = 4, /* run arguments differ from the plan's */
  GEMM_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed */
  GEMM_ERR_TIMEOUT = 6,       /* device: a pipeline wait exceeded its time limit */
  GEMM_ERR_BOUNDS = 7         /* device, bounds-checked build only: an index or copy
                                 coordinate failed its range check (the access was
                                 skipped; see gemm_check_t) */
} gemm_status_t;

typedef enum { GEMM_F16 = 0, GEMM_BF16 = 1 } gemm_dtype_t;

/* Epilogue applied to the fp32 accumulator before the output rounding:
 * GEMM_EPI_RELU is max(x, 0) (the Triton lecture notes' matmul example). */
typedef enum { GEMM_EPI_NONE = 0, GEMM_EPI_GELU_TANH = 1, GEMM_EPI_RELU = 2 } gemm_epilogue_t;

typedef enum {
  GEMM_PIPELINED = 0,     /* `stages`-deep ring, double-buffered accumulator */
  GEMM_SINGLE_BUFFER = 1  /* one ring slot, one accumulator (no overlap) */
} gemm_variant_t;

typedef struct gemm_plan gemm_plan_t; /* opaque */

/* Optional tuning knobs for gemm_plan_create_ex.  Zero means "choose". */
typedef struct {
  int tile_n;          /* output tile width: 0 (auto), 64, 128 or 256 */
  int raster_group;    /* tile rows walked together for L2 reuse; 0 = auto */
  int max_ctas;        /* cap on persistent CTAs; 0 = one per SM */
  int cta_group;       /* CTAs per output tile: 0 (auto), 1 (128-row tiles), or 2
                          (a CTA pair on two SMs computes a 256-row tile with
                          cta_group::2 MMAs; tile_n then 128 or 256) */
  int tail_split;      /* the last, partial wave of tiles: 0 = auto, -1 = off,
                          1 = stream-K (the last one to two waves' K iterations are
                          shared out evenly; a tile split between two CTAs is summed
                          in a fixed order, so results are deterministic),
                          k in {2, 3, 4} = cut each leftover tile along N into k
                          narrower tiles (>= 64 columns each, k must divide tile_n) */
  int64_t timeout_ns;  /* per-wait limit on the device; 0 = default (2 s), <0 = invalid */
  int b_kn;            /* 1: B is stored K x N (row-major, N contiguous, ldb = N), so
                          C = epi(A . B) -- the [M,K] @ [K,N] form of the Mosaic GPU
                          guide's Hopper example; 0 (default): B is N x K and
                          C = epi(A . B^T) */
  int out_f32;         /* 1: C is fp32 (4-byte elements, written unrounded from the fp32
                          accumulator after the epilogue), as in the Triton lecture notes'
                          matmul example; 0: C has the inputs' 16-bit type */
  int debug_fault;     /* test hook, 0 in normal use.  1: the first CTA's copy engine
                          never receives its first K slice, so the pipeline's waits run
                          out their time limit and gemm_plan_check reports
                          GEMM_ERR_TIMEOUT (every other tile still completes).
                          2 (bounds-checked build only; GEMM_ERR_INVALID_ARG in the
                          normal build): the range check of the first CTA's first copy
                          is made to fail -- its coordinates are valid -- so the copy is
                          skipped and gemm_plan_check reports GEMM_ERR_BOUNDS with
                          GEMM_CHECK_TMA_COORD */
  int k_serpentine;    /* K order of successive waves of tiles: 0 = auto (alternate when
                          the A and B rows one wave of tiles reads exceed half of L2),
                          1 = alternate (a CTA's odd-numbered tiles walk K downwards, so
                          the next wave starts on the slices the last one read most
                          recently), -1 = always upwards.  Ignored for a single row of
                          tiles, whose K loops are staggered instead */
  int epi_groups;      /* epilogue warps: 0 = auto (eight when K is at most 16 slices of 64
                          or the tiles form a single row, where the epilogue is not hidden
                          behind the main loop; else four), 1 = four (one per TMEM lane
                          quarter, two staging buffers each), 2 = eight (two per quarter,
                          each taking half of a tile's columns) */
} gemm_tuning_t;

/* Read-only description of what a plan will launch (for tests and benchmarks). */
typedef struct {
  int tile_m, tile_n, tile_k;  /* CTA output tile and K slice */
  int stages;                  /* ring depth actually used */
  int accumulators;            /* TMEM accumulator buffers (1 or 2) */
  int raster_group;
  int grid;                    /* persistent CTAs launched */
  int64_t num_tiles;
  size_t smem_bytes;           /* dynamic shared memory per CTA */
  int pads_operands;           /* last run staged A/B through padded scratch */
  int tma_store;               /* last run stored C with bulk tensor stores */
  int kernels_per_run;         /* kernel launches of the last run */
  int sm_count;
  int cta_group;               /* CTAs per output tile (1 or 2) */
  int64_t tail_tiles;          /* tiles of the last wave that are cut into narrow tiles */
  int tail_splits;             /* narrow tiles per cut tile (1 = none) */
  int64_t work_units;          /* whole tiles + narrow tiles walked by the CTAs */
  int stream_k;                /* 1: the tail_tiles are shared out stream-K */
  int out_f32;                 /* C is fp32 */
  int b_kn;                    /* B is stored K x N */
  int k_sub;                   /* K slices of tile_k per ring slot: stages / k_sub
                                  slots of k_sub slices each (same shared memory) */
  int host_panels;             /* blocks of C (row panels x column panels) gemm_run_host
                                  pipelines its copies in (0 before the first pipelined
                                  call) */
  int k_serpentine;            /* 1: successive waves alternate their K direction */
  int l2_prefetch_first;       /* 1: operands exceed 3/4 of L2, so each CTA prefetches its first
                                  ring's slices into L2 before waiting on the previous
                                  kernel in the stream */
  int sk_cluster;              /* 1: every tile is split into two K halves on the two CTAs
                                  of a cluster, whose partial sum moves through
                                  distributed shared memory */
  int epi_groups;              /* epilogue column groups: 1 (four warps) or 2 (eight) */
  int stream_k_first;          /* 1: each CTA takes its stream-K share before its whole tiles
                                  (chosen when stream-K is on and the serpentine K order off),
                                  so the fix-ups of shared tiles overlap later tiles; 0: the
                                  stream-K share comes last */
} gemm_plan_info_t;

/* Create a plan for C = epi(A . B^T) of the given sizes on `device`.
 * stages: ring depth >= 1 (GEMM_SINGLE_BUFFER requires 1).  With automatic
 * tiling the widest output tile whose ring fits the shared-memory budget is
 * chosen.  Returns GEMM_ERR_SMEM_BUDGET when even the narrowest tile does not
 * fit (never clamps `stages`).  On success *out owns device memory: release
 * it with gemm_plan_destroy.  On failure *out is set to NULL. */
gemm_status_t gemm_plan_create(gemm_plan_t** out, int64_t M, int64_t N, int64_t K,
                               gemm_dtype_t dtype, gemm_epilogue_t epi, int stages,
                               gemm_variant_t variant, int device);

/* As gemm_plan_create, with explicit tuning (tuning may be NULL). */
gemm_status_t gemm_plan_create_ex(gemm_plan_t** out, int64_t M, int64_t N, int64_t K,
                                  gemm_dtype_t dtype, gemm_epilogue_t epi, int stages,
                                  gemm_variant_t variant, int device,
                                  const gemm_tuning_t* tuning);

/* Enqueue C = epi(A . B^T) on `stream` (a cudaStream_t; NULL = legacy default
 * stream).  A, B, C: device pointers as described above; C must not overlap
 * A or B.  M, N, K, dtype, epi and stages must equal the plan's
 * (GEMM_ERR_PLAN_MISMATCH otherwise).  M == 0 or N == 0 is a no-op; K == 0
 * writes zeros (GELU(0) = 0).  Asynchronous: does not synchronise the
 * stream or the device.
 *
 * CUDA graphs: gemm_run and gemm_run_bias may be captured into a graph
 * (stream capture, any mode) and the graph replayed; each replay computes
 * the GEMM of the buffers' contents at that time.  A plan whose operands
 * need padded copies allocates that scratch in its first run (and again
 * when a later run needs more), so run such a plan once before capturing
 * it.  Consecutive GEMMs on one stream may be launched early (programmatic
 * dependent launch), but each waits for its predecessor's results before
 * reading memory, so one GEMM's C may be the next one's A or B. */
gemm_status_t gemm_run(gemm_plan_t* plan, const void* A, const void* B, void* C,
                       int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                       gemm_epilogue_t epi, int stages, void* stream);

/* As gemm_run, with a per-column bias:
 *   C[i,j] = epi(sum_k A[i,k] B[j,k] + bias[j]).
 * bias: device pointer to N values of `dtype` (2-byte aligned, not
 * overlapping C), or NULL for none (then the same as gemm_run).  The bias is
 * added to the fp32 accumulator, after any stream-K partial and before the
 * epilogue function.  With K == 0, C = epi(bias) in every row.
 *
 * The pages define no bias term.  This is the reading of a Linear layer's
 * bias (the GELU workload, Y = gelu(X . W^T), is such a layer): one value per
 * output feature, i.e. per column of C. */
gemm_status_t gemm_run_bias(gemm_plan_t* plan, const void* A, const void* B, const void* bias,
                            void* C, int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                            gemm_epilogue_t epi, int stages, void* stream);

/* End-to-end call with HOST buffers: copies hA (M*K) and hB (N*K) to
 * plan-owned device buffers, runs the GEMM on `stream`, copies C back to hC
 * (M*N) and synchronises `stream` before returning.  Pinned host memory gives
 * asynchronous copies; pageable memory works too.  The first call allocates
 * the device buffers.
 *
 * Problems with at least 32 MiB of copies and at least 2 blocks run in
 * blocks of C so that copies overlap the GEMM: 1-4 row panels of >= 1536 rows
 * (whole tiles), and -- for B stored N x K with K % 8 == 0 -- 1-4 column
 * panels of >= 1536 columns (multiples of 256; otherwise whole rows of C).
 * The panels of A and of B (rows of B for a column panel, else all of B)
 * come in on one plan-owned copy stream, alternating A0, B0, A1, B1, ..., and
 * each block's GEMM runs on `stream` as soon as its two panels are in,
 * through a block plan of its own.  The block of C goes back (a 2-D copy) on
 * a second copy stream while the next blocks compute.  The copy streams wait
 * for the work already queued on `stream`, and the call returns after all of
 * them finish.  gemm_plan_check also reports the block plans' device
 * status. */
gemm_status_t gemm_run_host(gemm_plan_t* plan, const void* hA, const void* hB, void* hC,
                            int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                            gemm_epilogue_t epi, int stages, void* stream);

/* Where a device-side wait ran out of time (the detail of GEMM_ERR_TIMEOUT):
 * role << 16 | wait id, role 1 = TMA producer, 2 = MMA issuer, 3 = epilogue. */
typedef enum {
  GEMM_WAIT_PRODUCER_EMPTY = (1 << 16) | 1, /* producer: a ring slot to become free */
  GEMM_WAIT_PRODUCER_DRAIN = (1 << 16) | 2, /* producer: its last copies to land */
  GEMM_WAIT_MMA_ACC_EMPTY = (2 << 16) | 1,  /* MMA issuer: the epilogue to free an accumulator */
  GEMM_WAIT_MMA_FULL = (2 << 16) | 2,       /* MMA issuer: a ring slot's copies */
  GEMM_WAIT_MMA_DRAIN = (2 << 16) | 3,      /* MMA issuer: its last MMAs to complete */
  GEMM_WAIT_EPI_FULL = (3 << 16) | 1,       /* epilogue: an accumulator to be filled */
  GEMM_WAIT_SK_FLAG = (3 << 16) | 2,        /* stream-K owner: the partner's partial */
  GEMM_WAIT_SK_COPY = (3 << 16) | 3,        /* stream-K owner: the partial's bytes */
  GEMM_WAIT_SK_FREE = (3 << 16) | 4         /* cluster split: the owner's ring to be free */
} gemm_wait_t;

/* Bounds-checked build.  The library can be compiled with
 * -DSPGEMM_BOUNDS_CHECKS=1 (the Python package builds it as
 * libspgemm_checked.so next to libspgemm.so).  Its kernels check, before each
 * access, the indexes and coordinates they derive: tile indexes, K slots and
 * copy coordinates (the K coordinate of a tiled copy must be 16-byte
 * aligned), TMEM columns, ring slots, staging buffers, C blocks and stream-K
 * workspace slots.  A failed check records GEMM_ERR_BOUNDS with the check's
 * identity (below) as the detail, skips the access and ends that role; the
 * other roles' bounded waits then run out, the kernel exits and the GPU stays
 * usable -- nothing traps.  This guards the shared-memory ring the Mosaic
 * GPU pipelining guide's delay_release discussion is about: a slot index or
 * coordinate that went wrong is reported instead of corrupting memory.  The
 * checks cost time; the normal build compiles them out.
 * Detail codes: role << 16 | 16 + id, role 0 = kernel set-up, 1 = TMA
 * producer, 2 = MMA issuer, 3 = epilogue. */
typedef enum {
  GEMM_CHECK_SMEM_LAYOUT = (0 << 16) | 16, /* ring + staging + barriers exceed the launch's
                                              shared memory */
  GEMM_CHECK_TILE = (1 << 16) | 16,        /* a unit's tile index or tile coordinates */
  GEMM_CHECK_K_SLICE = (1 << 16) | 17,     /* a K slot outside the unit's range or K */
  GEMM_CHECK_TMA_COORD = (1 << 16) | 18,   /* a copy coordinate out of range or unaligned */
  GEMM_CHECK_MMA_TMEM = (2 << 16) | 16,    /* accumulator columns beyond the TMEM allocation */
  GEMM_CHECK_MMA_SLOT = (2 << 16) | 17,    /* a ring slot index beyond the ring */
  GEMM_CHECK_EPI_TMEM = (3 << 16) | 16,    /* TMEM columns read beyond the allocation */
  GEMM_CHECK_STAGING = (3 << 16) | 17,     /* a staging buffer beyond the warp's area */
  GEMM_CHECK_STORE = (3 << 16) | 18,       /* a C block outside the tile grid or unaligned */
  GEMM_CHECK_PARTIAL = (3 << 16) | 19,     /* a stream-K workspace slot beyond the workspace */
  GEMM_CHECK_FIXUP = (3 << 16) | 20        /* a partial's shared-memory region beyond the ring */
} gemm_check_t;

/* 1 when this library is the bounds-checked build, 0 otherwise. */
int gemm_bounds_checked(void);

/* Synchronise the plan's device and read (then clear) its device status word.
 * *device_status receives GEMM_OK or the code a kernel recorded (e.g.
 * GEMM_ERR_TIMEOUT); *detail (may be NULL) receives the place it was recorded
 * (a gemm_wait_t, 0 with no error).  Returns GEMM_ERR_CUDA if the
 * synchronisation itself failed. */
gemm_status_t gemm_plan_check(gemm_plan_t* plan, int32_t* device_status, int32_t* detail);

/* Describe the plan's launch configuration. */
gemm_status_t gemm_plan_get_info(const gemm_plan_t* plan, gemm_plan_info_t* info);

/* ---- Planning without a plan ------------------------------------------------
 * None of the pages has a counterpart to these calls; they expose the
 * planner that gemm_plan_create runs, for capacity planning and for testing
 * it on a machine without a GPU.
 *
 * The properties of a device that the planner reads. */
typedef struct {
  int sm_count;       /* streaming multiprocessors (cudaDeviceProp::multiProcessorCount) */
  int smem_optin;     /* opt-in dynamic shared memory per block, bytes
                         (cudaDevAttrMaxSharedMemoryPerBlockOptin) */
  int64_t l2_bytes;   /* L2 cache size, bytes (cudaDeviceProp::l2CacheSize) */
  int pair_clusters;  /* 2-CTA clusters the CTA-pair kernels can keep resident at once
                         (cudaOccupancyMaxActiveClusters; every kernel runs one CTA per SM) */
} gemm_device_desc_t;

/* Fill *desc from `device`.  GEMM_ERR_UNSUPPORTED unless it is an sm_103
 * device; GEMM_ERR_CUDA if a query fails. */
gemm_status_t gemm_device_query(int device, gemm_device_desc_t* desc);

/* What gemm_plan_create_ex with these arguments would choose on a device
 * with the properties in *desc, written to *info exactly as
 * gemm_plan_get_info reports it for a plan that has not run yet (the fields
 * about the last run -- pads_operands, tma_store, kernels_per_run,
 * host_panels -- are 0).  Argument errors are the same as
 * gemm_plan_create_ex's, plus GEMM_ERR_INVALID_ARG for a NULL desc or info
 * or a description field out of range (sm_count, smem_optin < 1;
 * l2_bytes, pair_clusters < 0).  Makes no CUDA call, allocates nothing and
 * does not check the device's architecture. */
gemm_status_t gemm_plan_describe(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                                 gemm_epilogue_t epi, int stages, gemm_variant_t variant,
                                 const gemm_tuning_t* tuning, const gemm_device_desc_t* desc,
                                 gemm_plan_info_t* info);

/* Free everything the plan owns.  NULL is allowed.  Waits for the plan's
 * device work to finish first. */
void gemm_plan_destroy(gemm_plan_t* plan);

/* Static text for a status code ("GEMM_OK", ...). */
const char* gemm_status_string(gemm_status_t s);

/* Static text for the detail of a device status word: a gemm_wait_t ("MMA
 * issuer waiting for a ring slot's copies", ...) or a gemm_check_t ("copy
 * coordinate out of range or unaligned", ...); "" for 0, "unknown wait"
 * otherwise. */
const char* gemm_wait_detail_string(int32_t detail);

/* Last error message recorded by this host thread (argument that failed,
 * CUDA error text), or "" if none.  The pointer stays valid until the next
 * call into this library from the same thread. */
const char* gemm_last_error(void);

/* Shared-memory bytes of the operand ring, the TileLang tutorial's
 * shared_bytes(): stages * (bm*bk + bn*bk) * elem_bytes.  Returns 0 if an
 * argument is not positive. */
size_t gemm_smem_bytes(int bm, int bn, int bk, int elem_bytes, int stages);

/* Library version as "major.minor.patch". */
const char* gemm_version(void);

/* ---- Allocation-free entry point --------------------------------------------
 * None of the pages has a counterpart to this call; it exists for users of
 * the library, not for the method.
 *
 * For callers that cannot allocate device memory (no cudaMalloc, no
 * allocating library routine): code running under an allocator it does not
 * control, a runtime that forbids allocations once it has started, or a
 * caller that must not add allocations while other GPU work is being set
 * up.  gemm_run needs a plan, and a plan allocates its status word and,
 * for operands whose row pitch or base address is not 16-byte aligned,
 * scratch for padded copies.  gemm_run_noalloc takes no plan and allocates
 * nothing: its scratch is one static device array of
 * GEMM_NOALLOC_SCRATCH_BYTES (plus 256 bytes of status words) that every
 * GPU loading this library reserves until the process exits.
 *
 * Arguments: as gemm_run, without the plan; A, B, C are device pointers on
 * the current device, `stream` a cudaStream_t (NULL = legacy stream).
 * Asynchronous.  Returns GEMM_ERR_INVALID_ARG when the padded copies would
 * need more than GEMM_NOALLOC_SCRATCH_BYTES (that is, when
 * ((A misaligned or K % 8 ? M : 0) + (B misaligned or K % 8 ? N : 0)) *
 * round_up(K, 8) * 2 exceeds it); aligned problems need no scratch and have
 * no such limit.  Device-side wait timeouts are recorded in the static
 * status word but not reported (there is no plan to read them from).
 *
 * The first call on each device sets that device up (takes the device
 * address of the static array with cudaGetSymbolAddress, sets the kernels'
 * shared-memory limits, looks up the tensor-map encoder).  Make that first
 * call before any stream capture.  A set-up that fails is not kept: the
 * call returns its error and the next call on that device tries again.  Every call on a device shares the one
 * array and leaves its contents behind (the status words are cleared at the
 * start of each call): calls whose work overlaps on the GPU -- on different
 * streams, or from different host threads -- race on it. */
#define GEMM_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

gemm_status_t gemm_run_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N,
                               int64_t K, gemm_dtype_t dtype, gemm_epilogue_t epi, int stages,
                               void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPGEMM_GEMM_H_ */
