/*
 * tgemm.h -- C ABI of the software-pipelined tiled GEMM for GB300 (sm_103a).
 *
 * The operation.  C[M,N] = A[M,K] . B[N,K]^T with fp16 or bf16 operands,
 * fp32 accumulation, and C either fp32 (the raw accumulator) or the operand
 * dtype (fp32 rounded to nearest even).  This is the tiled GEMM of the
 * TileLang tutorial, chapter 11 "Pipeline and autotuning": section 1.1 gives
 * the tiled body (per output tile, clear an fp32 accumulator, loop over K in
 * block_K steps copying an A tile and a B tile into shared memory and
 * multiplying with transpose_B), section 3.5 gives the kernel signature
 * (A:(M,K), B:(N,K), C:(M,N); tile block_M x block_N x block_K; num_stages),
 * and section 2.3 / 4.4 give the pipelining: num_stages copies of each
 * operand tile, slot ko % num_stages, so that loads of k-block ko+1.. overlap
 * the math of k-block ko.
 *
 * Memory.  Every matrix is dense and row-major: A is M x K (K contiguous),
 * B is N x K (K contiguous), C is M x N (N contiguous).  Device pointers are
 * owned by the caller and must be 16-byte aligned; the library never
 * allocates or frees them.  The row pitch of every matrix must be a multiple
 * of 16 bytes (K % 8 == 0; N % 4 == 0 for fp32 C, N % 8 == 0 for 16-bit C),
 * as the tensor-memory-access engine requires.
 *
 * Errors.  Every function returns a tgemm_status_code (0 = TGEMM_OK) or a
 * value documented below; nothing throws across this boundary and nothing
 * aborts the process.  Arguments are checked before anything is launched.
 *
 * Threads and streams.  A plan may be used from one host thread at a time.
 * Different plans are independent.  Launches of one plan on different streams
 * may overlap, except with split_k > 1: those share the plan's workspace, so
 * they must be ordered (one stream, or events between them).
 */
#ifndef TGEMM_H
#define TGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (the same object as cudaStream_t / CUstream); NULL is
 * the legacy default stream. */
typedef struct CUstream_st *tgemm_stream_t;

/* Opaque plan: validated shape, tile, depth and launch configuration. */
typedef struct tgemm_plan_s *tgemm_plan_t;

enum tgemm_dtype {
    TGEMM_F16 = 0,  /* IEEE binary16 */
    TGEMM_BF16 = 1, /* bfloat16 */
    TGEMM_F32 = 2   /* IEEE binary32, output only */
};

enum tgemm_status_code {
    TGEMM_OK = 0,
    TGEMM_ERR_INVALID_ARG = 1,       /* a size, pointer or config outside its documented range */
    TGEMM_ERR_UNSUPPORTED_DTYPE = 2, /* dtype not F16/BF16, or out_dtype not F32/dtype */
    TGEMM_ERR_ALIGNMENT = 3,         /* pointer or row pitch not a multiple of 16 bytes */
    TGEMM_ERR_SMEM_BUDGET = 4,       /* tile x num_stages does not fit in shared memory */
    TGEMM_ERR_NO_KERNEL = 5,         /* tile shape the kernel does not implement */
    TGEMM_ERR_ARCH = 6,              /* current device is not compute capability 10.3 */
    TGEMM_ERR_CUDA = 7,              /* a CUDA runtime or driver call failed */
    TGEMM_ERR_TIMEOUT = 8,           /* a pipeline wait inside the kernel ran out of time */
    TGEMM_ERR_CHECK = 9              /* an internal bounds or alignment check failed; only a
                                        build with TGEMM_DEBUG_CHECKS=1 makes these checks */
};

/*
 * Shared-memory upper bound of the pipeline, in bytes: num_stages copies of
 * one A tile (block_M x block_K) and one B tile (block_K x block_N), times the
 * element size of dtype.  Chapter 11, section 4.5 ("multi-buffering and the
 * on-chip capacity limit").  Returns -TGEMM_ERR_UNSUPPORTED_DTYPE or
 * -TGEMM_ERR_INVALID_ARG (negative) on bad input.  Host only; needs no GPU.
 */
int64_t tgemm_smem_bound(int dtype, int block_M, int block_N, int block_K, int num_stages);

/*
 * Dynamic shared memory the kernel actually requests for this config, in
 * bytes: the pipeline ring (the bound above, each slot aligned for the
 * swizzled layout), the output staging buffers, the ring's full/empty
 * barriers, the accumulator barriers and alignment slack.  Negative status
 * on bad input, as above.  Host only.
 */
int64_t tgemm_smem_bytes(int dtype, int out_dtype, int block_M, int block_N, int block_K,
                         int num_stages);

/*
 * Per-block shared-memory limit (cudaDevAttrMaxSharedMemoryPerBlockOptin) of
 * the current device, in bytes; negative status if no device can be queried.
 */
int tgemm_smem_limit(void);

/*
 * Validate a problem and config against a given per-block shared-memory
 * limit, without touching a GPU: the same checks tgemm_plan makes, in the
 * same order, with `smem_limit` standing in for the queried device limit.
 *   - dtype in {F16, BF16}, out_dtype in {F32, dtype}     -> UNSUPPORTED_DTYPE
 *   - M, N >= 0, K >= 0, each <= 2^31 - 257 (a coordinate
 *     rounded up to a whole tile stays a 32-bit TMA
 *     coordinate); num_stages >= 1; at most 2^30 output
 *     tiles (times K splits)                               -> INVALID_ARG
 *   - K % 8 == 0, N * out_bytes % 16 == 0 (row pitch)      -> ALIGNMENT
 *   - block_M in {64, 128, 256} (64: M = 64 tensor-core
 *     instructions; cta_pair: 256 only); block_N a multiple
 *     of 32 in [32, 256] (with cta_pair up to 512);
 *     block_K in {16, 32, 64, 128} (16-bit
 *     operands: rows of 32, 64 or 128 bytes, or two 128-byte
 *     K-panels for 128)                                     -> NO_KERNEL
 *   - tgemm_smem_bound > smem_limit or
 *     tgemm_smem_bytes > smem_limit                         -> SMEM_BUDGET
 * The budget rule is the one of chapter 11 sections 4.5 and 5.1: a config
 * over budget is rejected before anything is launched, rather than failing
 * at launch.  M == 0 or N == 0 is a valid empty product; K == 0 is a valid
 * empty reduction (C is all zeros).
 */
int tgemm_validate(int64_t M, int64_t N, int64_t K, int dtype, int out_dtype, int block_M,
                   int block_N, int block_K, int num_stages, int64_t smem_limit);

/*
 * Create a plan on the current CUDA device.  Runs tgemm_validate with the
 * device's queried limit, checks that the device is sm_103 (ERR_ARCH),
 * allocates a 16-byte device status word owned by the plan, and sets the
 * kernel's dynamic shared-memory attribute.  On success *out is a plan owned
 * by the caller (free it with tgemm_destroy); on failure *out is NULL.  The
 * pages' analogue is matmul(M, N, K, block_M, block_N, block_K, num_stages,
 * ...) of chapter 11 section 3.5; its `threads` argument has no counterpart
 * because the kernel's warp roles fix the block at 352 threads (two TMA
 * producer warps, one for A and one for B, an MMA warp and eight epilogue
 * warps).
 */
int tgemm_plan(tgemm_plan_t *out, int64_t M, int64_t N, int64_t K, int dtype, int out_dtype,
               int block_M, int block_N, int block_K, int num_stages);

/*
 * Options of tgemm_plan_ex (zero-initialise, then set what you need).
 *   cta_pair: 0 = one CTA per output tile (tgemm_plan's behaviour).  1 = pairs
 *     of CTAs (thread-block clusters of 2) on neighbouring SMs share each
 *     block_M = 256 tile: one M = 256 tensor-core instruction per K step spans
 *     both SMs, each CTA holds 128 rows of A, block_N / 2 rows of B and 128
 *     rows of the accumulator.  Only block_M = 256 is accepted.  block_N may
 *     then also be a multiple of 32 from 288 to 512: two N = block_N / 2
 *     instructions per K step share the A operand (each SM pulls less operand data per FLOP, but
 *     the accumulator fills tensor memory, so the epilogue of a tile no longer
 *     overlaps the next tile's K loop).  Each CTA is a
 *     block in the sense of the pages' budget rule: the bound checked is
 *     num_stages x (128 x block_K + block_K x block_N / 2) x element size.
 *   group_m: M-tiles per raster group of the persistent schedule (0: 8).
 *   split_k: 0 or 1 = no split.  s > 1 = split the K loop of every tile into
 *     s ranges of whole k-blocks (fewer if K has fewer k-blocks), computed as
 *     separate work units that write fp32 partial tiles to a workspace of
 *     s x ceil(M / block_M) x block_M x N floats the plan allocates.  Then
 *     the partials are added in split order (0, 1, ..., s-1) and rounded once
 *     to C's type: by a second kernel, or with grid_reduce = 1 by the same
 *     kernel after a grid-wide barrier.  Both give the same bits.
 *     The order of every sum depends only on the tile shape and s, never on
 *     num_stages, so results stay bit-identical across depths.  For long K
 *     and few output tiles (more SMs than tiles).  At most 64, and the
 *     workspace rows, s x ceil(M / block_M) x block_M, below 2^31
 *     (32-bit TMA coordinates); else INVALID_ARG.
 *   prefetch: 0 = num_stages.  1 <= D <= num_stages = the producer issues the
 *     loads of k-block i only after the MMAs of k-block i - D have finished,
 *     i.e. it runs at most D k-blocks ahead whatever the number of buffers.
 *     This separates the pipeline depth from the buffer count the way the
 *     pages separate a manual schedule's max(stage) + 1 from num_stages
 *     (chapter 11 sections 3.3 and 4.4): D = 1 serialises load and compute,
 *     D = 2 is the two-stage schedule of matmul_manual.  Results do not
 *     depend on D.
 *   cluster_k: 0 or 1 = split K reduces through the workspace and a second
 *     kernel, as above.  c = 2, 4 or 8 = the kernel reduces the splits itself:
 *     one CTA per (tile, split) work unit, launched as thread-block clusters
 *     of c CTAs that take c consecutive splits of one tile.  A cluster adds
 *     its c partial accumulators through distributed shared memory, in rank
 *     order; when split_k / c clusters share a tile, each writes its fp32 sum
 *     to a workspace of (split_k / c) x ceil(M / 128) x 128 x N floats, and
 *     the last to finish adds them in cluster order and writes C.  The order
 *     of every sum depends only on the tile shape, split_k and c, so results
 *     stay bit-identical across num_stages (they differ in rounding from the
 *     two-kernel reduction, whose order is sequential).  Requires cta_pair = 0,
 *     block_M = 128, an effective split count that is a multiple of c,
 *     block_N / c a multiple of 32, and num_stages x (A + B slot) of at least
 *     128 x block_N x 4 bytes (the exchanged partials land in the operand
 *     ring); else INVALID_ARG (SMEM_BUDGET for the ring).  Launches of one such
 *     plan must be ordered (one stream, or events between them): they share
 *     the workspace and the arrival counters.
 *   stream_operands: 0 = plain operand loads.  1 = the operand loads carry an
 *     L2 evict-first hint: when L2 needs room, lines of A and B go before other
 *     data (for instance dirty lines, whose eviction costs a write to HBM).
 *     It pays when each operand line is read once, or by a few tiles at about
 *     the same time (long K over few tiles); it costs where tiles of later
 *     waves read the same rows again (large square problems).  Results do not
 *     depend on it.  Other values: INVALID_ARG.
 *   stream_k: 0 = every tile is one persistent work unit.  1 = when the tiles
 *     do not fill the last wave of workers (CTAs, or CTA pairs), the tiles
 *     past the last whole wave are shared out by k-blocks: each worker takes
 *     an equal contiguous run of the tail's k-block iterations, tile after
 *     tile, so all workers finish together.  A tile covered by several runs is
 *     finished by the last of them to complete: each run stores its fp32
 *     partial to a workspace the plan allocates (workers x 2 x block_M x
 *     block_N floats) and counts in; the last adds the runs' partials in k
 *     order and writes C.  No CTA waits for another.  Sums stay in a fixed
 *     order (a function of the shape, the tile and the number of workers),
 *     so results are bit-identical across num_stages.  Not combined with
 *     split_k > 1 or cluster_k > 1 (INVALID_ARG).  Left off (no tail) when the
 *     tiles fill whole waves or the tail has fewer than two k-blocks per
 *     worker.  Launches of one such plan must be ordered.  On GB300 it does
 *     not pay yet: each lane of the epilogue holds one row, so the pieces'
 *     fp32 stores and the finishing loads touch 32 rows per instruction, and
 *     that traffic costs more than the idle tail it removes (8192^3 bf16:
 *     614 us against 598 us without it; 588 us with the piece traffic
 *     switched off in a probe).
 *   grid_reduce: with split_k > 1 and cluster_k <= 1: 0 = a second kernel
 *     reduces the K splits; 1 = the GEMM kernel does, after a grid-wide
 *     barrier.  The launch is then cooperative, so every CTA of the
 *     persistent grid is resident at once, and the barrier's wait is bounded
 *     by the watchdog.  Same results; no second launch, but on GB300 the
 *     512 x 512 x 32768 case measured 33 us against 31.5 us with the second
 *     kernel: reading the partials costs the same either way and the barrier
 *     adds its own wait.  Other values: INVALID_ARG.
 *   multicast_b: 0 = each CTA pair loads its own B rows.  1 = thread-block
 *     clusters of four CTAs, two pairs that take the two M-adjacent tiles of
 *     one N-block (the second pair's tile lies past M when the M-blocks are
 *     odd in number; it loads zeros and stores nothing).  The CTAs of rank r
 *     and r ^ 2 hold the same rows of B: each loads one part of them and TMA
 *     multicast writes it into both, so each SM issues the copies of half its
 *     B rows and L2 serves each B line once per cluster.  A slot is refilled
 *     once both pairs' MMAs have finished with it.  Same MMAs in the same
 *     order: results are bit-identical to cta_pair alone.  Requires
 *     cta_pair = 1, no K split, stream_k, grid_reduce or cluster_k, and a
 *     CTA's B box (block_N / 2, or block_N / 4 for a tile wider than 256) of
 *     at least 16 rows (parts of whole 8-row swizzle atoms); else INVALID_ARG.
 *     Clusters of four fit fewer at a time than pairs (36 on GB300, 144 SMs).
 *     On GB300 it pays where B's rows straddle L2 lines: 4000 x 3000 x 5000
 *     fp16 (a 10,000-byte row pitch) ran 83.4-83.9 us against 88.1-88.6 us
 *     with pairs alone.  4096^3 and 8192^3 ran slower with it (their tiles
 *     fill rounds of 36 clusters poorly).
 */
typedef struct tgemm_plan_opts {
    int cta_pair;
    int group_m;
    int split_k;
    int prefetch;
    int cluster_k;
    int stream_operands;
    int grid_reduce;
    int stream_k;
    int multicast_b;
} tgemm_plan_opts;

/* tgemm_validate with options (NULL = defaults): the option ranges above
 * (cta_pair 0 or 1, group_m 0..4096, split_k 0..64, prefetch 0..num_stages,
 * cluster_k 0, 1, 2, 4 or 8, stream_operands, grid_reduce and stream_k 0 or 1;
 * stream_k with split_k > 1 or cluster_k > 1) give INVALID_ARG, then the checks of
 * tgemm_validate, the split-K workspace rule and the cluster_k rules, as
 * tgemm_plan_ex makes them. */
int tgemm_validate_ex(int64_t M, int64_t N, int64_t K, int dtype, int out_dtype, int block_M,
                      int block_N, int block_K, int num_stages, int64_t smem_limit,
                      const tgemm_plan_opts *opts);

/* tgemm_plan with options (NULL = defaults); ERR_INVALID_ARG for an option out
 * of range, ERR_NO_KERNEL for cta_pair with block_M != 256. */
int tgemm_plan_ex(tgemm_plan_t *out, int64_t M, int64_t N, int64_t K, int dtype, int out_dtype,
                  int block_M, int block_N, int block_K, int num_stages, const tgemm_plan_opts *opts);

/*
 * Enqueue C = A . B^T on `stream`.  A, B, C are device pointers with the
 * layouts above (16-byte aligned, caller-owned; C must not overlap A or B).
 * Returns after the launch is enqueued; results are ready when the stream
 * has run it.  The pages' analogue is kernel(A, B, C) with C the output.
 * ERR_INVALID_ARG for a NULL plan or pointer (unless the product is empty),
 * ERR_ALIGNMENT for a misaligned pointer, ERR_CUDA if the launch fails.
 */
int tgemm_run(tgemm_plan_t plan, const void *A, const void *B, void *C, tgemm_stream_t stream);

/*
 * End-to-end form of tgemm_run for operands in host memory: enqueue on
 * `stream` the copies hA -> dA and hB -> dB, the GEMM into dC, and the copy
 * dC -> hC.  hA/hB/hC are host buffers of the same layouts (page-locked
 * memory makes the copies asynchronous); dA/dB/dC are caller-owned device
 * buffers of the same sizes.  The library allocates nothing.  Returns after
 * enqueueing; hC is valid once the stream has run.  Errors as tgemm_run.
 */
int tgemm_run_host(tgemm_plan_t plan, const void *hA, const void *hB, void *hC, void *dA,
                   void *dB, void *dC, tgemm_stream_t stream);

/*
 * Read and clear the plan's device status word.  Call after the stream that
 * ran the plan has been synchronised (this call itself synchronises through
 * a blocking copy).  Returns TGEMM_OK, or TGEMM_ERR_TIMEOUT if a pipeline
 * wait in any CTA ran past the watchdog limit (the kernel then stops its
 * pipeline, waits for its copies in flight, frees its tensor memory and
 * returns instead of hanging; C is undefined).  Negative ERR_CUDA on a failed
 * copy.  `detail` (may be NULL) receives 4 ints: code, warp role (0 producer,
 * 1 MMA, 2 epilogue), block index, and the pipeline iteration that timed out.
 * For a plan with cluster_k > 1, a status other than TGEMM_OK also zeroes the
 * plan's arrival counters, which a launch that gave up may have left part-way.
 */
int tgemm_status(tgemm_plan_t plan, int *detail);

/*
 * Watchdog limit of every in-kernel pipeline wait, in nanoseconds of
 * %globaltimer (default 2e9, or the environment variable TGEMM_WATCHDOG_NS
 * read at plan time).  0 restores the default.
 */
int tgemm_set_watchdog_ns(tgemm_plan_t plan, uint64_t ns);

/*
 * Test hook: when `on` is nonzero, the MMA warp of every CTA waits, at its
 * first k-block, on a barrier that nothing arrives on, so that the watchdog
 * path runs (status TGEMM_ERR_TIMEOUT).  No fault, trap or hang results.
 */
int tgemm_debug_stall(tgemm_plan_t plan, int on);

/* Launch geometry and resources of a plan (for reports and the sweep). */
typedef struct tgemm_plan_info {
    int64_t M, N, K;
    int dtype, out_dtype, block_M, block_N, block_K, num_stages;
    int tiles_m, tiles_n, num_tiles, grid, threads;
    int num_k_blocks;    /* ceil(K / block_K) */
    int acc_stages;      /* accumulator buffers in tensor memory (1 or 2) */
    int tmem_columns;    /* tensor-memory columns allocated per CTA */
    int64_t smem_bytes;  /* dynamic shared memory requested per CTA */
    int64_t smem_bound;  /* the pages' num_stages * (A + B tile) bound */
    int smem_limit;      /* device per-block limit at plan time */
    int num_sms;
    int cta_pair;        /* 1: clusters of two CTAs share each tile */
    int split_k;         /* effective K splits (1: none) */
    int num_units;       /* persistent work units: tiles x K splits (multicast_b: pairs of tiles) */
    int prefetch;        /* producer lead in k-blocks */
    int cluster_k;       /* > 1: K splits reduced in the kernel by clusters of this many CTAs */
    int stream_operands; /* 1: operand loads carry an L2 evict-first hint */
    int grid_reduce;     /* 1: K splits reduced in the GEMM kernel after a grid-wide barrier */
    int stream_k_tiles;  /* tiles of the stream-K tail (0: none) */
    int multicast_b;     /* 1: clusters of two CTA pairs share B through TMA multicast */
} tgemm_plan_info;

int tgemm_get_plan_info(tgemm_plan_t plan, tgemm_plan_info *info);

/*
 * Allocation-free form of tgemm_plan + tgemm_run (+ tgemm_status), for callers
 * that cannot allocate device memory: code running where cudaMalloc is
 * unavailable or must not be called (a custom allocator's own hooks, a service
 * that fixes its device footprint at start-up, a runtime that hands the library
 * only the buffers it works on).  The tutorial pages have no counterpart; this
 * is an interface addition of this library.
 *
 * Arguments and checks are those of tgemm_plan and tgemm_run (same status
 * codes; sizes, dtypes, tiles and depths they reject are rejected here).  The
 * kernel's only memory besides A, B and C is its 16-byte status record; here it
 * lives in a fixed 256-byte array inside the library's CUDA module, which every
 * GPU that loads the library holds until the process exits.  The record always
 * fits that array (the library checks this when it is compiled), so no size of
 * problem needs more.  The call allocates nothing: no cudaMalloc, no cudaFree,
 * no allocating library routine.
 *
 * The call enqueues on `stream` a clear of the array's status record and the
 * kernel.  If `status` is non-NULL it then copies the record back, waits for
 * `stream`, and stores TGEMM_OK or TGEMM_ERR_TIMEOUT there (or TGEMM_ERR_CHECK
 * from a build with TGEMM_DEBUG_CHECKS=1); if NULL the call returns right after
 * enqueueing.  Waiting for the stream is not allowed while it is being
 * captured, so on a capturing stream a non-NULL `status` is rejected with
 * TGEMM_ERR_INVALID_ARG before anything is enqueued.  All calls on a device
 * share the one array: calls whose kernels overlap on the same GPU (for
 * instance on two streams) race on it, and the status they report is then
 * unreliable.
 *
 * Every call looks up the array's device address for the current device (a
 * host-side lookup that allocates nothing), so a reset device or a new
 * context is handled.  The first call on each device makes the runtime load
 * the library's module there and sets the kernel's shared-memory ceiling for
 * that device; make that first call before any stream capture.
 */
int tgemm_run_noalloc(int64_t M, int64_t N, int64_t K, int dtype, int out_dtype, int block_M, int block_N,
                      int block_K, int num_stages, const void *A, const void *B, void *C, tgemm_stream_t stream,
                      int *status);

/* Free a plan, its status word and its split-K workspace.  The device memory
 * goes back through cudaFree, which first waits for the device to finish its
 * work, so launches of the plan still in flight complete before it is freed.
 * NULL is accepted (no-op). */
int tgemm_destroy(tgemm_plan_t plan);

/* Static text for a status code (never NULL). */
const char *tgemm_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* TGEMM_H */
