/*
 * tmagemm.h -- C ABI of the GB300 (sm_103a) TMA-pipelined fp16 GEMM.
 *
 * Operation ("GEMM II -- pipelining with TMA", Step 4: the A tile is loaded at
 * {m, k} and the B tile at {n, k}, each BLK x BLK_K, fp16; the baseline
 * paragraph: fp32 accumulate; the TMA-store epilogue: the accumulator is
 * narrowed to the output dtype):
 *
 *     C[m][n] = sum_{k < K} A[m][k] * B[n][k]
 *
 *   A : M x K fp16, row-major (element (m,k) at A[m*K + k])
 *   B : N x K fp16, row-major, i.e. B^T is K-major (element (n,k) at B[n*K + k])
 *   C : M x N, row-major (ldc = N), fp32 or fp16 (round to nearest even)
 *   accumulation in fp32 on the tensor cores.
 *
 * Everything runs on one GPU, in the library's own CUDA kernels; there is no
 * CPU fallback: calls fail with an error code when no device is present.
 *
 * Threading: plans are independent; one plan must not be used by two host
 * threads at once.  Errors: every function that can fail returns a gemm_status
 * (or NULL) and leaves a message for gemm_last_error() (thread-local).
 */
#ifndef TMAGEMM_H
#define TMAGEMM_H

#include <stdint.h>

#if defined(__GNUC__)
#define TMAGEMM_API __attribute__((visibility("default")))
#else
#define TMAGEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gemm_plan gemm_plan; /* opaque; owned by the library */

typedef enum { GEMM_OUT_F32 = 0, GEMM_OUT_F16 = 1 } gemm_dtype;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1, /* NULL pointer, non-positive size, bad option value */
    GEMM_ERR_UNSUPPORTED = 2, /* shape/alignment the TMA path cannot take, or a
                                 stage count that does not fit shared memory */
    GEMM_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
    GEMM_ERR_TIMEOUT = 4,     /* a kernel wait exceeded its bound (see
                                 gemm_get_device_status) */
    GEMM_ERR_NO_DEVICE = 5    /* no usable CUDA device / wrong architecture */
} gemm_status;

/* Kernel variants: the ablation ladder of "GEMM II -- pipelining with TMA"
 * (Steps 3-6) plus the warp-specialised forms. */
typedef enum {
    GEMM_VAR_AUTO = 0,              /* CTA pairs when M > 128 and there are at
                                       least (SM count / 2) 256x128 tiles --
                                       GEMM_VAR_DYNAMIC_2CTA, or
                                       GEMM_VAR_PERSISTENT_2CTA when the options
                                       set grid or stream_k = 2 -- else
                                       GEMM_VAR_PERSISTENT */
    GEMM_VAR_SYNC_TILED = 1,        /* Step 3: thread copies, one MMA at a time */
    GEMM_VAR_TMA_SERIAL = 2,        /* Step 4: TMA load + expect_tx, serial loop */
    GEMM_VAR_PIPELINED = 3,         /* Step 5: PIPE_DEPTH ring, lock-step prefetch */
    GEMM_VAR_WS_PIPELINED = 4,      /* producer warp / MMA warp / epilogue warps,
                                       full+empty ring, one tile per CTA */
    GEMM_VAR_PERSISTENT = 5,        /* warp-specialised, grid = SM count, grouped
                                       raster, two TMEM accumulators */
    GEMM_VAR_PERSISTENT_LOCKSTEP = 6, /* Step 6 as printed: persistent CTAs running
                                       the lock-step Step-5 loop */
    GEMM_VAR_PERSISTENT_2CTA = 7,   /* warp-specialised, persistent, on CTA pairs
                                       (clusters of 2): 256 x block_n tiles with
                                       tcgen05.mma.cta_group::2, each CTA loading
                                       its own half of the operands; block_n 128,
                                       160, 192, 224 or 256, chosen by wave
                                       efficiency */
    GEMM_VAR_DYNAMIC_2CTA = 8,      /* the CTA-pair kernel with a dynamic tile
                                       schedule ("GEMM II -- pipelining with
                                       TMA", Step 6: cluster launch control as
                                       the upgrade of the static assignment):
                                       the grid has one cluster per tile, and
                                       a running cluster cancels clusters that
                                       have not started
                                       (clusterlaunchcontrol.try_cancel) and
                                       computes their tiles.  grid must be 0;
                                       stream_k = 2 splits the tail instead
                                       (see stream_k); gemm_schedule_unit
                                       reports only each cluster's own unit,
                                       the rest being assigned at run time */
} gemm_variant;

/* Plan options; a zero field means "choose automatically". */
typedef struct {
    int variant;        /* gemm_variant */
    int pipe_depth;     /* shared-memory stages, 1..8 (ring variants) */
    int block_n;        /* output tile width: 64, 128 or 256 (tile height 128);
                           for the CTA-pair variant see GEMM_VAR_PERSISTENT_2CTA */
    int group_m;        /* raster group height in M tiles (default 16 for CTA
                           pairs, 8 otherwise) */
    int grid;           /* persistent variants: CTAs to launch (default: SM count) */
    int wait_budget_ms; /* bound on any single in-kernel wait (default 2000) */
    int debug_stall;    /* 1: the producer first waits on a barrier that nothing
                           completes, so the run ends in GEMM_ERR_TIMEOUT (for
                           testing the watchdog; warp-specialised variants) */
    int stream_k;       /* persistent warp-specialised variants: 0 = auto (off),
                           1 = off, 2 = on whenever the tile count leaves a
                           partial last wave.  With stream-K the tiles of the
                           partial last wave are split into K-block ranges
                           shared evenly by all CTAs (or pairs); partial sums go
                           through a workspace the plan owns and are added in a
                           fixed order, so results do not vary from run to run.
                           GEMM_VAR_DYNAMIC_2CTA with stream_k = 2: the tiles of
                           the partial last wave (all tiles when there are fewer
                           than SM count / 2) are each split into S = 2..4 equal
                           K ranges, S = (SM count / 2) / those tiles, each
                           range at least 4 stages, run as separate units;
                           gemm_config.sk_max_contrib is S. */
    int l2_policy;      /* L2 eviction priority of the operand loads (warp-specialised
                           variants): 0 = default, 1 = A evict_last and B
                           evict_first, 2 = A evict_first and B evict_last,
                           3 = both evict_last */
    int k_order;        /* persistent warp-specialised variants: 0 = auto (snake),
                           1 = every tile walks K upwards, 2 = "snake": a CTA walks K
                           downwards on every other tile, so each tile starts on
                           the A slices its predecessor (the previous wave of
                           the same raster group) used last and that are still
                           in L2 */
    int block_k;        /* K extent of one pipeline stage: 64 = one 128-byte
                           swizzle atom (64 fp16); 128 or 256 = two or four
                           atoms per stage ("05 Async Data Movement - TMA",
                           Using 3D TMA to Move Multiple Swizzle Atoms), loaded
                           as that many boxes per operand and consumed by 8 or
                           16 MMAs behind one barrier round trip.  128: the
                           warp-specialised variants (CTA pairs and single
                           CTAs); 256: the single-CTA warp-specialised variants
                           (persistent, ws_pipelined).  pipe_depth then counts
                           stages of this extent, and stream-K splits K in such
                           stages.  A block of the last stage past K arrives
                           zero-filled and is skipped.  0 = auto: 128 for the
                           CTA-pair variants when K is a multiple of 64
                           (128-byte aligned operand rows) and pipe_depth is
                           not set, else 64 */
} gemm_options;

/* Resolved configuration of a plan (also returned by gemm_select_config). */
typedef struct {
    int variant;
    int block_m, block_n, block_k;
    int pipe_depth;
    int group_m;
    int grid;           /* CTAs launched */
    int threads;        /* threads per CTA */
    int tiles_m, tiles_n, num_tiles, k_blocks;
    int smem_bytes;     /* dynamic shared memory per CTA */
    int tmem_cols;      /* TMEM columns allocated per CTA */
    int tx_bytes;       /* bytes one stage's barrier expects (A + B tile) */
    int dp_tiles;       /* tiles computed whole */
    int sk_tiles;       /* tiles of the stream-K part (0: none) */
    int sk_kb_per_worker; /* pipeline stages (of block_k) of the stream-K part
                             per CTA / pair */
    int sk_max_contrib; /* most CTAs / pairs that share one stream-K tile */
    long long workspace_bytes; /* device workspace the plan allocates for stream-K */
    int a_rows;         /* rows of A per stage: 128, or 64 when M <= 64 (single-CTA
                           warp-specialised variants; the MMA still computes 128
                           rows and rows past M are never stored) */
    int tail_halves;    /* GEMM_VAR_DYNAMIC_2CTA, automatic (stream_k = 0) with
                           256-column tiles and stages of K = 128: when all the
                           tiles fit in at most half the resident clusters (SM
                           count / 4), each is computed as two 256 x 128 tiles
                           by two clusters (no partial sums to combine); this
                           is the number of tiles so split, 0 = none.  The grid
                           is 2 x (num_tiles + tail_halves) CTAs */
} gemm_config;

/* Create a plan for C[M x N] = A[M x K] . B[N x K]^T on the current CUDA
 * device.  dtype_out is a gemm_dtype.  Preconditions: M, N, K >= 1 and
 * < 2^31; K % 8 == 0 and N * sizeof(out) % 16 == 0 (TMA global strides are
 * multiples of 16 bytes, "05 Async Data Movement - TMA", the tensor-map
 * descriptor; a TMA copy must start on a 16-byte boundary).  Returns NULL on
 * error (gemm_last_status() / gemm_last_error() say why).  The plan owns host
 * state, a 32-byte device status record and, when its configuration uses
 * stream-K, a device workspace of gemm_config.workspace_bytes; because of
 * that workspace, runs of one plan must not overlap on the GPU (use one plan
 * per concurrent stream).
 * Passage: "GEMM II -- pipelining with TMA", Steps 5 and 6 -- what is fixed
 * before the launch (PIPE_DEPTH stages sized against shared memory, the tile
 * shape, a grid of one CTA per SM) -- and "B200 Tma Pipeline Designer",
 * Execution, steps 2 (the tensor-map descriptor of each operand) and 6 (the
 * stage ring and its shared-memory total against residency). */
TMAGEMM_API gemm_plan* gemm_create_plan(int64_t M, int64_t N, int64_t K, int dtype_out);

/* Same with options (NULL = all automatic).  An explicit pipe_depth whose ring
 * does not fit in shared memory fails with GEMM_ERR_UNSUPPORTED.
 * Passage: "GEMM II -- pipelining with TMA", Steps 3-6 (the variants of the
 * ablation ladder) and Step 5 (PIPE_DEPTH); tilus matmul-hopper v2,
 * Multi-Stage Software Pipelining (deeper rings force smaller tiles). */
TMAGEMM_API gemm_plan* gemm_create_plan_ex(int64_t M, int64_t N, int64_t K, int dtype_out,
                               const gemm_options* opts);

/* Enqueue C = A . B^T on `cuda_stream` (a cudaStream_t; NULL = legacy default
 * stream).  A, B, C are DEVICE pointers owned by the caller, 16-byte aligned,
 * laid out as above; C's rows and columns beyond M x N are never written.
 * Asynchronous: returns after the launch.  Argument and launch errors are
 * returned at once; an in-kernel timeout is reported by
 * gemm_get_device_status after the caller has synchronised the stream.  The
 * plan must be used on the device it was created on.
 *
 * Dependent launch: the warp-specialised variants (everything but the
 * lock-step ladder) are launched as programmatic dependents of the work before
 * them on the stream.  Their CTAs may become resident and set up shared memory
 * and TMEM while the previous kernel drains, but they read A and B and write C
 * only after all earlier work on the stream has completed (griddepcontrol.wait
 * before the first global-memory access), so stream order is kept.  After
 * set-up they allow the next launch on the stream to be scheduled early; a
 * kernel launched after this one as a programmatic dependent must itself wait
 * (griddepcontrol.wait) before reading C.
 *
 * CUDA graphs: the launch may be captured into a graph once the plan has run
 * once outside the capture (that first run sets the kernel's shared-memory
 * limit).  A replay repeats the captured run counter, so after a timeout in
 * one replay the later replays of that graph end as aborted too: capture
 * again.  Plans with stream-K tiles (stream_k = 2 and a partial last wave)
 * have fix-up tickets keyed by the run counter, which a replay would repeat
 * and so leave shared tiles unwritten: the static schedule refuses capture
 * with GEMM_ERR_UNSUPPORTED, and a captured launch of the dynamic schedule
 * runs every tile whole.
 * Passage: "GEMM II -- pipelining with TMA", Steps 4-6 (one elected thread
 * issues the bulk-tensor loads and announces their bytes; the staged
 * mainloop; the TMA-store epilogue), on tensor maps encoded for the pointer
 * triple ("05 Async Data Movement - TMA", How One Thread Describes an Entire
 * Tile). */
TMAGEMM_API int gemm_run(gemm_plan* plan, const void* A, const void* B, void* C, void* cuda_stream);

/* End-to-end variant of gemm_run for HOST buffers: copies A and B to device
 * buffers owned by the plan (allocated on first use, reused after), runs the
 * GEMM, copies C back and synchronises `cuda_stream`.  A, B, C are host
 * pointers.  When all three are page-locked and M >= 2048, the round trip is
 * pipelined in bands of rows: B and then A band by band go in on a copy
 * stream, each band's GEMM runs on `cuda_stream` (through a sub-plan per band)
 * as soon as its rows of A have landed, and each band of C comes back on a
 * second copy stream while later bands compute; otherwise the copies and the
 * GEMM run one after the other on `cuda_stream`.  Returns GEMM_ERR_TIMEOUT if
 * a kernel's watchdog fired.
 * Passage: none -- the pages define no interface, so this call belongs to the library's own boundary; the GEMM it runs is gemm_run's. */
TMAGEMM_API int gemm_run_host(gemm_plan* plan, const void* A, const void* B, void* C, void* cuda_stream);

/* Read (and clear) the plan's device status record.  Call after
 * synchronising the stream(s) the plan ran on.  Returns GEMM_OK or
 * GEMM_ERR_TIMEOUT (a wait ran past wait_budget_ms; the kernel then skipped
 * its remaining work, freed TMEM and exited, so C is incomplete), or
 * GEMM_ERR_CUDA if the read itself failed.
 * Passage: none -- the pages define no interface, so this call belongs to the library's own boundary.  The pages' barrier waits are unbounded ("05 Async
 * Data Movement - TMA", How to Wait for a TMA Load); the bound on each wait
 * and this record of where one ran out are the library's own. */
TMAGEMM_API int gemm_get_device_status(gemm_plan* plan);

/* Free the plan and the device memory it owns (NULL is allowed).  The caller
 * must have synchronised every stream the plan ran on.
 * Passage: none -- the pages define no interface, so this call belongs to the library's own boundary. */
TMAGEMM_API void gemm_destroy(gemm_plan* plan);

/* Message / code of the last failing call on this host thread (thread-local;
 * the message is empty after a call that succeeded).
 * Passage: none -- the pages define no interface, so this call belongs to the library's own boundary. */
TMAGEMM_API const char* gemm_last_error(void);
TMAGEMM_API int gemm_last_status(void);

/* Human-readable one-line description of the plan (variant, tile, depth,
 * shared memory, grid).  The string is owned by the plan.
 * Passage: none -- the pages define no interface, so this call belongs to the library's own boundary; the values it reports are the choices of "GEMM II
 * -- pipelining with TMA", Steps 5 and 6 (PIPE_DEPTH, tile, grid). */
TMAGEMM_API const char* gemm_plan_describe(const gemm_plan* plan);

/* The plan's resolved configuration.
 * Passage: none -- the pages define no interface, so this call belongs to the library's own boundary; see gemm_config for the pages' quantities it holds. */
TMAGEMM_API int gemm_plan_config(const gemm_plan* plan, gemm_config* out);

/* Record a device timeline of the following runs of `plan` into
 * `device_buffer` (caller-owned device memory of at least
 * grid * (units_per_cta + 1) * 10 uint64 words, 8-byte aligned), or stop
 * recording (NULL).  For each CTA, record 0 is a header {start ns, end ns, SM
 * id, units processed} and records 1..units_per_cta hold, per work unit, the
 * globaltimer stamps of its milestones: {tile << 32 | K blocks, first load
 * issued, last load issued, accumulator free, first MMA issued, last MMA
 * issued and committed, accumulator complete at the epilogue, last store
 * issued, ns the MMA issuer waited for loaded stages, ns the producer waited
 * for free stages}.  These are the prologue / steady-state / drain phases of the stage
 * ring ("GEMM II -- pipelining with TMA", the pipeline Gantt: TMA and MMA
 * lanes; "B200 Tma Pipeline Designer", the three-phase timeline).
 * Warp-specialised variants only; a few stores per unit. */
TMAGEMM_API int gemm_set_trace(gemm_plan* plan, void* device_buffer, int units_per_cta);

/* ---- host-only helpers (no GPU needed; used by tests and tools) ---- */

/* Resolve options into a configuration for a device with `sm_count` SMs and
 * `smem_optin` bytes of opt-in shared memory per block, exactly as
 * gemm_create_plan_ex does.  Returns a gemm_status.
 * Passage: as gemm_create_plan_ex; the stage-count limit is "B200 Tma
 * Pipeline Designer", Execution, step 6 (total shared memory of the ring
 * against residency). */
TMAGEMM_API int gemm_select_config(int64_t M, int64_t N, int64_t K, int dtype_out, const gemm_options* opts,
                       int sm_count, int smem_optin, gemm_config* out);

/* Output tile (m_tile, n_tile) of linear tile index `tile` in the grouped
 * raster order the kernels use ("GEMM II -- pipelining with TMA", Step 6,
 * l2_group_size).  Returns GEMM_ERR_INVALID_ARG if tile is out of range. */
TMAGEMM_API int gemm_schedule_tile(const gemm_config* cfg, int64_t tile, int* m_tile, int* n_tile);

/* Work unit `index` (0, 1, ...) of persistent worker `worker` (a CTA, or a
 * CTA pair for the pair variants) under `cfg`, in the order the kernels
 * process them: whole tiles first, then the worker's share of the stream-K
 * part.  Under the dynamic schedule only the worker's own unit (index 0) is
 * fixed before the run -- the rest are taken by cancellation while the
 * kernel runs.  Writes
 * the tile (raster index), its K-block range [kb0, kb1) and the worker's rank
 * among the tile's contributors; returns 1, or 0 when the worker has no unit
 * `index`, or GEMM_ERR_INVALID_ARG.
 * Passage: "GEMM II -- pipelining with TMA", Step 6 (each persistent CTA
 * walks its own sequence of tiles); the split of K among workers (stream-K)
 * has no passage. */
TMAGEMM_API int gemm_schedule_unit(const gemm_config* cfg, int worker, int index, int* tile,
                                   int* kb0, int* kb1, int* contrib, int* ncontrib);

/* Byte offset of logical byte `byte_in_row` of row `row` inside a
 * 1024-byte-aligned tile of 128-byte rows stored with the 128-byte swizzle
 * ("05 Async Data Movement - TMA", "How TMA Writes a Swizzled Layout"), as
 * the thread-copy variant writes it and the TMA engine lays it out. */
TMAGEMM_API int64_t gemm_sw128_offset(int64_t row, int64_t byte_in_row);

/* Allocation-free variant of gemm_create_plan + gemm_run + gemm_destroy for
 * callers that cannot call cudaMalloc: processes whose device memory is
 * owned by a framework's caching allocator or a pre-reserved arena (a foreign
 * cudaMalloc fails or is forbidden there), and latency-critical loops that
 * cannot pay the device synchronisation that cudaMalloc/cudaFree imply.  The
 * pages have no counterpart of this entry point.
 *
 * Runs the kernel the automatic plan of gemm_create_plan(M, N, K, dtype_out)
 * runs for C = A . B^T -- the dynamic CTA-pair kernel for large problems, the
 * single-CTA persistent kernel for small or skinny ones; automatic plans never
 * use stream-K, the only option that needs a workspace -- with the same
 * operands, layouts, preconditions and arithmetic as gemm_run, on
 * `cuda_stream`.  It allocates nothing: its only scratch memory, the kernel's
 * 32-byte watchdog status record, lives in a file-scope device array of 256
 * bytes (the stated maximum; a build whose record outgrew it would be rejected
 * with GEMM_ERR_UNSUPPORTED) that every GPU loading this library holds until
 * the process exits.  It calls no cudaMalloc, cudaFree or allocating library
 * routine.
 *
 * Set-up: the first call on each device looks up that array's device address
 * (cudaGetSymbolAddress, with that device current), and so does the first
 * call after the current context has changed (a cudaDeviceReset by the
 * caller, or a context the caller made current): an address looked up in a
 * destroyed context is never used.  Make such a first call before any stream
 * capture begins.  Every call on a device shares the one array and clears it
 * at the start (an asynchronous memset on `cuda_stream`), so calls that
 * overlap on the GPU race on the status record: serialise them.
 *
 * device_status: non-NULL makes the call synchronise `cuda_stream` and store
 * GEMM_OK or GEMM_ERR_TIMEOUT there, which is also returned.  NULL makes the
 * call asynchronous like gemm_run, and then a watchdog timeout is not
 * reported at all: no call reads the shared record later, and the next call
 * clears it.  Callers that must know whether C is complete pass
 * device_status. */
TMAGEMM_API int gemm_run_noalloc(int64_t M, int64_t N, int64_t K, int dtype_out, const void* A,
                                 const void* B, void* C, void* cuda_stream, int* device_status);

#ifdef __cplusplus
}
#endif

#endif /* TMAGEMM_H */
