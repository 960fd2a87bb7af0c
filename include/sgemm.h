/*
 * sgemm.h -- C ABI of the GB300 FP32 SGEMM library (libsgemm_gb300.so).
 *
 * The operation (all entry points): C = alpha * A * B + beta * C on
 * row-major float32 matrices, A is M x K, B is K x N, C is M x N; element
 * [i][j] of a matrix with leading dimension ld sits at base + i*ld + j.
 *   -- "How a Matmul Kernel Gets Fast", section 1 "The problem, and what
 *      cuBLAS is" (GEMM is C = alpha*A*B + beta*C);
 *   -- "Learn: Optimizing GEMM", section 3 "Rung 0 -- Naive (recap)" (the
 *      row-major layout and one output as a length-K dot product scaled by
 *      alpha, plus beta times the old C).
 *
 * Arithmetic: IEEE float32 fused multiply-adds on the CUDA cores, each
 * output summed in ascending k unless the plan's description says
 * "k_order=split" (a split-K plan adds fixed-order partial sums).  The
 * epilogue is out = alpha*acc (beta == 0) or fmaf(alpha, acc, beta*C_old).
 *
 * One variant computes differently and is never picked by the shape table:
 * "tf32x3_128x256x32_s2" (sgemm_plan_with_config or SGEMM_FORCE_CONFIG).
 *   - Operation: the same C = alpha*A*B + beta*C on the tensor cores.
 *   - Method: each operand is split as x = hi + lo into two TF32 values (round to
 *     nearest; |x - hi - lo| <= 2^-22 |x|), and the product is
 *     hi*hi + hi*lo + lo*hi accumulated in float32 (k_order=tf32x3).
 *   - Accuracy: results stay within the acceptance bound
 *     |C - C_ref| <= 4 K 2^-24 |A||B| + 1e-6. The plan refuses K < 16 with
 *     SGEMM_ERR_UNSUPPORTED.
 *   - Limits: it needs finite inputs below about 2^127 in magnitude, where
 *     the split cannot overflow.
 *   - Memory: the plan allocates 2 (M + N) round_up(K, 4) floats for the split
 *     operands.
 *   - Launches: each run launches three kernels (two splits, then the GEMM).
 *   - Layout: any alignment and leading dimension are accepted.
 *
 * Conventions (BLAS readings where the pages are silent):
 *   - lda >= max(1, K), ldb >= max(1, N), ldc >= max(1, N), else
 *     SGEMM_ERR_INVALID_ARG.  Dimensions above 2^31 - 1, leading
 *     dimensions above 2^40, and a stored matrix (or strided batch of them)
 *     spanning more than 2^40 elements from its first to its last element
 *     give SGEMM_ERR_UNSUPPORTED: no device holds such a buffer.
 *   - M == 0 or N == 0: nothing is launched, SGEMM_OK.
 *   - K == 0 or alpha == 0: C = beta * C; A and B are not read.
 *   - beta == 0: C is not read (NaN or garbage in C does not propagate).
 *   - C must not share its address span (first to last element, rows and
 *     padding included) with A or B: sgemm_run returns
 *     SGEMM_ERR_UNSUPPORTED when they meet. A and B may overlap each other.
 *   - Any alignment and any leading dimension is accepted.  Fast paths
 *     need A and B 16-byte aligned with lda % 4 == 0 and ldb % 4 == 0; other
 *     inputs run a GPU kernel with scalar loads (there is no CPU path).
 *
 * Memory and threads: A, B and C are DEVICE pointers owned by the caller,
 * on the device that was current when the plan was made.  sgemm_run only
 * enqueues work on `stream` (a cudaStream_t; NULL is the legacy default
 * stream) and returns; results are ready when the stream reaches that point.
 * A plan is immutable after sgemm_plan returns and may be used from several
 * host threads.  No entry point allocates device memory inside sgemm_run.
 * sgemm_run only encodes tensor maps on the host and launches, so it can be
 * captured into a CUDA graph once the plan has run once outside capture.
 * A replayed stream-K launch stays correct: the CTA that consumes a partial
 * tile clears that tile's flag, so every run leaves the flags at zero.
 * A plan whose description says streamk=1 owns a device workspace (one
 * partial tile and one flag per CTA of its grid), allocated by sgemm_plan
 * and freed by sgemm_plan_destroy; so does a matrix-vector plan (kind=gemv)
 * with split > 1 (its partial sums).  Two runs of such a plan must not overlap
 * in time (same stream, or streams ordered by events), since both would
 * write the same workspace.  Every other plan may run on several streams
 * at once.
 *
 * Errors: every entry point returns a status and never aborts.  Launch
 * failures map to SGEMM_ERR_CUDA.  Faults during execution surface at the
 * caller's next synchronisation, as with any CUDA launch.  Every wait inside
 * a kernel has a time limit (default 4 s, raised for long products; see
 * sgemm_set_wait_timeout_ns);
 * a wait that runs out records SGEMM_ERR_TIMEOUT in a per-device status
 * word that sgemm_device_status reads.
 */
#ifndef SGEMM_GB300_H
#define SGEMM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct sgemm_plan_s *sgemm_plan_t;

typedef enum {
    SGEMM_OK = 0,
    SGEMM_ERR_INVALID_ARG = -1,  /* bad dimension, leading dimension, pointer or id */
    SGEMM_ERR_UNSUPPORTED = -2,  /* valid but outside what this build handles */
    SGEMM_ERR_CUDA = -3,         /* a CUDA runtime or driver call failed */
    SGEMM_ERR_TIMEOUT = -4,      /* a kernel wait ran past its time limit */
    SGEMM_ERR_NOMEM = -5,        /* host allocation failed */
    SGEMM_ERR_BOUNDS = -6        /* checked build only: a kernel index failed its bounds check */
} sgemm_status_t;

/*
 * Make a plan for one problem shape on the current device: validates the
 * dimensions, picks a kernel variant from the per-shape config table
 * (measured on GB300) and prepares it.  Allocates host memory, plus a
 * device workspace of grid * tile_m * tile_n floats and grid flags
 * (cudaMalloc) when the choice splits the last, partial wave of tiles --
 * or, with fewer tiles than CTA slots, every tile -- along K across the
 * whole grid (stream-K; describe reports streamk=1).
 * That workspace makes the sum order along K for the tail tiles a fixed
 * split: results stay bit-identical from run to run.
 * For M <= 4 the table picks the matrix-vector kernels (kind=gemv,
 * gemv_4x512), and for one product of 5 <= M <= 16 rows with B as stored
 * and at least 2^22 elements of B, the sixteen-row ones (gemv_16x1024,
 * which stream B through per-warp cp.async rings in shared memory): B is
 * streamed once, K is cut into chunks that fill whole waves of the GPU,
 * and with more than one chunk (split > 1) the plan owns a workspace of
 * batch x split x M x N floats (N rounded up to 4) whose partial sums a
 * second kernel adds in an order fixed by the shape (bit-identical runs);
 * that kernel is launched as a programmatic dependent of the first.
 * These kernels take any alignment and leading dimension, so such plans are
 * never repacked ("Writing a Fast Matmul in CUDA", "Why decode doesn't
 * care": a matrix-vector product uses each weight once and is bound by
 * memory bandwidth).
 * From M*N*K >= 2^24 on, an operand whose leading dimension is not a
 * multiple of 4 (rows that are not 16-byte multiples, which TMA cannot
 * read) gets a plan-owned copy with padded rows (cudaMalloc, M x K or
 * K x N floats); each run first copies it there with one kernel on the
 * run's stream, and describe reports repack=1 (A), 2 (B) or 3.  Runs of such a plan must not overlap
 * in time.
 * The environment variable SGEMM_FORCE_CONFIG=<variant name> overrides the
 * table choice (and then nothing is repacked).  *out is set only on SGEMM_OK.
 */
sgemm_status_t sgemm_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                          sgemm_plan_t *out);

/*
 * As sgemm_plan, but with variant `config_id` (0 .. sgemm_num_configs()-1)
 * instead of the table's choice.  SGEMM_ERR_UNSUPPORTED if that variant
 * cannot run this shape (for example a skinny-M variant with large M).
 */
sgemm_status_t sgemm_plan_with_config(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                      int64_t ldc, int config_id, sgemm_plan_t *out);

/* Flags for sgemm_plan_autotune. */
enum { SGEMM_TUNE_TENSOR_CORES = 1 };

/*
 * Autotuning: time every variant that takes this shape and return a plan
 * for the fastest. The pages autotune the kernel's tile parameters by
 * compiling every legal configuration, running it and keeping the winner
 * ("How a Matmul Kernel Gets Fast", the autotuning step). Here the compiled
 * configurations are this build's variants.
 *
 * Arguments:
 *   - A, B, C: scratch device buffers of the plan's shape and leading
 *     dimensions. C is overwritten (the timing runs use alpha = 1,
 *     beta = 0).
 *   - flags: SGEMM_TUNE_TENSOR_CORES also tries the split-TF32
 *     tensor-core variants, which compute differently (see above). By
 *     default only the FP32 FFMA variants compete.
 *   - times_ms: if not NULL, receives sgemm_num_configs() entries, the mean
 *     time per run of each variant (-1 where a variant was not tried).
 *   - stream: the stream the timing runs go on.
 *
 * Timing: each variant gets one warm run, then 5 runs back to back timed
 * with CUDA events on `stream`. L2 is not flushed between runs, so operands
 * that fit in L2 stay hot.
 *
 * Cache: winners are cached per (device, shape, leading dimensions,
 * flags). A later call with times_ms == NULL returns the cached choice
 * without timing.
 *
 * Behaviour: synchronous (it waits for the timing runs).
 *
 * Errors: as sgemm_plan. SGEMM_ERR_UNSUPPORTED if no variant could run.
 * M, N or K of 0 gives the table's plan without timing.
 */
sgemm_status_t sgemm_plan_autotune(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                   const float *A, const float *B, float *C, int flags, void *stream,
                                   double *times_ms, sgemm_plan_t *out);

/*
 * Plan a strided batch of `batch` independent products of one shape:
 * C_z = alpha * A_z * B_z + beta * C_z, z = 0 .. batch-1, with
 * A_z = A + z*stride_a, B_z = B + z*stride_b, C_z = C + z*stride_c (in floats),
 * all row-major with the leading dimensions of sgemm_plan. Run it with
 * sgemm_run (or sgemm_run_host) on the base pointers.
 *
 * Argument rules:
 *   - A and B may be shared between products (stride 0).
 *   - The C matrices must not overlap: stride_c >= (M-1)*ldc + N when
 *     batch > 1, else SGEMM_ERR_INVALID_ARG.
 *   - batch == 0 is a valid empty plan.
 *   - batch > 65535 gives SGEMM_ERR_UNSUPPORTED.
 *   - config_id: -1 for the table, else a variant id. Variants that do not
 *     run batches refuse batch > 1 with SGEMM_ERR_UNSUPPORTED.
 *
 * How it runs:
 *   - Every product of the batch runs in one launch.
 *   - For M <= 4 the matrix-vector kernels, the batch on their third grid
 *     dimension; they take any strides.
 *   - Transposed-A kernels, and for 4 < M <= 16 the stream-K few-row kernel:
 *     3-D tensor maps, batch outermost. They need stride_a and stride_b to
 *     be multiples of 4 that either do not overlap the matrices or are 0
 *     (one operand shared by every product); their grid and stream-K split
 *     span the whole batch.
 *   - Otherwise the scalar-load kernel runs, the batch on its third grid
 *     dimension.
 *
 * The pages do not batch; this is the BLAS-style strided batch. Many
 * products of one shape, two per attention head (Q K^T, then the scores
 * times V), are the motivating case in "CUDA Matrix Multiplication
 * Optimization: From Naive to Near-cuBLAS", "What This Means for Deep
 * Learning".
 */
sgemm_status_t sgemm_plan_batched(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                  int64_t batch, int64_t stride_a, int64_t stride_b, int64_t stride_c, int config_id,
                                  sgemm_plan_t *out);

/* Storage order and operand transposition for sgemm_plan_ex. */
enum { SGEMM_ROW_MAJOR = 0, SGEMM_COL_MAJOR = 1 };
enum { SGEMM_NO_TRANS = 0, SGEMM_TRANS = 1 };

/*
 * Plan C = alpha * op(A) * op(B) + beta * C for any storage order and
 * transposition (the BLAS SGEMM interface): op(A) is M x K, op(B) is K x N,
 * C is M x N.
 *   - order: SGEMM_ROW_MAJOR or SGEMM_COL_MAJOR, for all three matrices.
 *   - transa: A is stored M x K (SGEMM_NO_TRANS) or K x M (SGEMM_TRANS).
 *     transb: B is stored K x N or N x K.
 *   - lda, ldb, ldc: the distance between consecutive rows (row-major) or
 *     columns (column-major) of the stored matrices. Each must be at least
 *     that matrix's row length (row-major) or column length (column-major),
 *     and at least 1; otherwise SGEMM_ERR_INVALID_ARG.
 *   - config_id: -1 for the shape table, else a variant id as for
 *     sgemm_plan_with_config.
 *
 * sgemm_run and sgemm_run_host take A, B and C as stored.
 *
 * How it runs:
 *   - A column-major product runs as the row-major product
 *     C^T = op(B)^T op(A)^T over the same memory.
 *   - The FFMA kernels read row-major operands stored untransposed. A
 *     transposed operand is first transposed on the GPU into a buffer the
 *     plan allocates (cudaMalloc), one extra kernel per run -- except in
 *     the two native cases below.
 *   - The transposed-A kernels (tmat_*) read the product's A given
 *     transposed (row-major transa, or column-major transb: stored K x M)
 *     as stored, when its leading dimension is a multiple of 4.
 *   - The split-TF32 variant reads either layout directly. So does the
 *     few-row stream-K kernel for B given transposed (stored N x K, the
 *     usual weight layout of decode) when ldb is a multiple of 4, and the
 *     M <= 4 kernels for any ldb.  (The 5-to-16-row matrix-vector kernels
 *     read B only as stored, so with B given transposed the table keeps
 *     the few-row stream-K kernel for those rows.)
 *   - A plan that reads a transposed operand natively needs A and B 16-byte
 *     aligned at run time, else SGEMM_ERR_UNSUPPORTED (the M <= 4 kernels
 *     excepted: they take any alignment).
 * Runs of a plan with such a buffer must not overlap in time.
 *
 * The pages cover the row-major, untransposed product only; the other
 * layouts follow the BLAS SGEMM conventions. cuBLAS's layout coverage is
 * noted in "Writing a Fast Matmul in CUDA", "What cuBLAS and CUTLASS add".
 */
sgemm_status_t sgemm_plan_ex(int order, int transa, int transb, int64_t M, int64_t N, int64_t K, int64_t lda,
                             int64_t ldb, int64_t ldc, int config_id, sgemm_plan_t *out);

/*
 * sgemm_plan_ex for a strided batch: C_z = alpha * op(A_z) * op(B_z) + beta * C_z,
 * z = 0 .. batch-1, every operand stored in `order` (with transa / transb as
 * in sgemm_plan_ex) and the products stride_a / stride_b / stride_c floats
 * apart (0: one A or B shared by every product).  Run it with sgemm_run on
 * the base pointers.
 *
 * Argument rules: those of sgemm_plan_ex and sgemm_plan_batched; the C
 * matrices must not overlap (stride_c at least one stored C, else
 * SGEMM_ERR_INVALID_ARG).
 *
 * How it runs: as sgemm_plan_ex over the whole batch in one launch
 * (column-major swaps the operands and their strides).  A transposed
 * operand is read as stored where a kernel can (the product's A by the
 * transposed-A kernels when the product has more than 16 rows, the
 * product's B by the few-row kernels otherwise; leading dimension a multiple
 * of 4, or any for M <= 4); otherwise every product's operand is
 * transposed first into a plan buffer (batch times the operand; one for a
 * shared operand).  The split-TF32 variants do not run batches.  Runs of a
 * plan must not overlap in time.
 *
 * The pages neither batch nor transpose; this combines the BLAS SGEMM
 * conventions of sgemm_plan_ex with the strided batch of sgemm_plan_batched.
 * Attention (two products per head, S = Q K^T then O = P V) is the
 * motivating case in "CUDA Matrix Multiplication Optimization: From Naive
 * to Near-cuBLAS", "What This Means for Deep Learning".
 */
sgemm_status_t sgemm_plan_ex_batched(int order, int transa, int transb, int64_t M, int64_t N, int64_t K,
                                     int64_t lda, int64_t ldb, int64_t ldc, int64_t batch, int64_t stride_a,
                                     int64_t stride_b, int64_t stride_c, int config_id, sgemm_plan_t *out);

/*
 * Enqueue C = alpha*A*B + beta*C on `stream` (a cudaStream_t, may be NULL).
 * A, B, C are device pointers with the plan's shape and leading dimensions.
 * A and B may be NULL only when K == 0 or alpha == 0; C may be NULL only
 * when M == 0 or N == 0.  If A or B is not 16-byte aligned, a variant that
 * needs alignment falls back to the scalar-load kernel for this call.
 */
sgemm_status_t sgemm_run(sgemm_plan_t plan, float alpha, const float *A, const float *B, float beta,
                         float *C, void *stream);

/*
 * The same product from HOST buffers: copies hA and hB (and hC when
 * beta != 0) into the caller's device buffers dA, dB, dC with
 * cudaMemcpyAsync, runs sgemm_run on them, and copies dC back into hC, all
 * on `stream`; returns after enqueueing (synchronise the stream before
 * reading hC).  Host matrices are dense with the plan's leading
 * dimensions.  Pinned host memory makes the copies asynchronous.
 */
sgemm_status_t sgemm_run_host(sgemm_plan_t plan, float alpha, const float *hA, const float *hB,
                              float beta, float *hC, float *dA, float *dB, float *dC, void *stream);

/*
 * A stream of `count` products of the plan's shape from HOST memory:
 * product i reads hA[i], hB[i] (and hC[i] when beta != 0) and writes hC[i].
 *
 * Buffers: dA, dB, dC each point to TWO device buffers of the plan's size,
 * owned by the caller. Products alternate between the two sets.
 *
 * Overlap: while product i computes on `stream`, the inputs of product i+1
 * copy in on one stream and the result of product i-1 copies out on
 * another, so the copies run under the kernels. The two copy streams and
 * six events belong to the plan, made on the first call (no device memory
 * is allocated).
 *
 * Returns after enqueueing. Once `stream` reaches this point, every result
 * is in host memory. Host memory should be pinned for the copies to be
 * asynchronous.
 *
 * Concurrency: calls on one plan must not overlap in time.
 *
 * Errors: as sgemm_run_host. SGEMM_ERR_INVALID_ARG for count < 0 or a
 * missing pointer.
 *
 * The pages time kernels only; this entry exists for end-to-end use.
 */
sgemm_status_t sgemm_run_host_pipelined(sgemm_plan_t plan, int count, float alpha, const float *const *hA,
                                        const float *const *hB, float beta, float *const *hC, float *const *dA,
                                        float *const *dB, float *const *dC, void *stream);

/* Free a plan and its device workspace, if any (the device that was
 * current at sgemm_plan must be current here).  NULL is accepted. */
sgemm_status_t sgemm_plan_destroy(sgemm_plan_t plan);

/*
 * Write a one-line description of the plan's choice into buf (at most n
 * bytes, NUL-terminated): variant name, tile sizes, grid, k order.
 */
sgemm_status_t sgemm_plan_describe(sgemm_plan_t plan, char *buf, size_t n);

/* Number of kernel launches one sgemm_run of this plan makes (into *out). */
sgemm_status_t sgemm_plan_launches(sgemm_plan_t plan, int *out);

/* The chosen variant's id (into *out). */
sgemm_status_t sgemm_plan_config_id(sgemm_plan_t plan, int *out);

/* Number of kernel variants in this build, and the name of one. */
int sgemm_num_configs(void);
const char *sgemm_config_name(int config_id);

/* Static text for a status code. */
const char *sgemm_status_string(sgemm_status_t status);

/*
 * Read (and with reset != 0, clear) the current device's kernel status
 * word.  Synchronises the device.  Returns SGEMM_OK, SGEMM_ERR_TIMEOUT if a
 * kernel wait ran out since the last reset, SGEMM_ERR_BOUNDS if (in the
 * checked build, libsgemm_gb300_checked.so, compiled with -DSGEMM_CHECKED)
 * a kernel's shared-memory or workspace index failed its bounds check and
 * the access was skipped, or SGEMM_ERR_CUDA.
 */
sgemm_status_t sgemm_device_status(int reset);

/*
 * Time limit, in nanoseconds, for every wait inside the library's kernels
 * on later launches (process-wide; default 4e9).  0 restores the default.
 * A launch never gets less than a floor that grows with its work: the time
 * the whole product (2*M*N*K*batch FLOPs) would take at 1e10 FLOP/s per SM,
 * about 1/45 of the rate the FFMA kernels sustain on GB300.  A stream-K
 * finisher's wait for its contributors can legitimately last as long as
 * their K-ranges, so the floor keeps long problems clear of the limit
 * (4096^3: 0.09 s, below the 4 s default; 65536^3 on 152 SMs: 370 s).
 */
sgemm_status_t sgemm_set_wait_timeout_ns(uint64_t timeout_ns);

/*
 * The wait limit a launch of an M x N x K product (over `batch` products)
 * gets on a device with num_sms SMs: the larger of the current setting and
 * that work-based floor.  Pure host arithmetic, no CUDA call.  *out is set
 * on SGEMM_OK; negative sizes, num_sms < 1 or out == NULL give
 * SGEMM_ERR_INVALID_ARG.  (An operational aid; the pages have no
 * counterpart.)
 */
sgemm_status_t sgemm_wait_limit_ns(int64_t M, int64_t N, int64_t K, int64_t batch, int num_sms, uint64_t *out);

/*
 * The variant the shape table picks for a row-major, untransposed product
 * (M x K times K x N, leading dimensions lda and ldb; `batch` products with
 * element strides stride_a and stride_b, 0 = shared, when batch > 1) on a
 * device with num_sms SMs -- the choice sgemm_plan / sgemm_plan_batched make
 * for that device.  b_trans != 0: B is given transposed (stored N x K), as
 * sgemm_plan_ex passes it.  `name` (name_size bytes, caller-owned) receives
 * the variant's name; *repack_a / *repack_b (either may be NULL) are set to
 * 1 when the plan would first copy that operand into rows padded to 16
 * bytes.  Pure host arithmetic, no CUDA call.  Invalid sizes or leading
 * dimensions, num_sms < 1, or a name buffer too small give
 * SGEMM_ERR_INVALID_ARG.  (An introspection aid; the per-shape choice
 * follows "How a Matmul Kernel Gets Fast": configurations measured per shape
 * class.)
 */
sgemm_status_t sgemm_table_choice(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t batch,
                                  int64_t stride_a, int64_t stride_b, int b_trans, int num_sms, char *name,
                                  size_t name_size, int *repack_a, int *repack_b);

/*
 * The persistent grid a transposed-A plan uses for `tiles` C tiles of
 * k_slices 32-deep k-slices each, with ctas_per_sm CTAs of the variant
 * resident on each of num_sms SMs ("Writing a Fast Matmul in CUDA, Step by
 * Step", "Size effects" and "What cuBLAS and CUTLASS add": a partial last
 * wave split along K).  *grid = CTAs launched; *dp_waves = whole waves of
 * tiles run data-parallel first; *sk_iters = k-slices of the remaining tiles
 * shared out over the grid (0: no split).  Whenever *sk_iters > 0 it is at
 * least *grid, so every CTA holds at least one slice.  Pure host arithmetic,
 * no CUDA call; negative counts, num_sms < 1, ctas_per_sm < 1 or a NULL
 * output give SGEMM_ERR_INVALID_ARG.
 */
sgemm_status_t sgemm_streamk_schedule(int64_t tiles, int64_t k_slices, int num_sms, int ctas_per_sm, int64_t *grid,
                                      int *dp_waves, int64_t *sk_iters);

/*
 * Self-test of the wait limit: launches one thread that waits, with limit
 * timeout_ns, on a barrier phase that nothing completes, then synchronises
 * the stream.  Returns SGEMM_ERR_TIMEOUT (and clears the status word) when
 * the wait gave up as designed; SGEMM_OK would mean the wait never ran out.
 */
sgemm_status_t sgemm_selftest_wait_timeout(uint64_t timeout_ns, void *stream);

/*
 * Size of the static scratch used by sgemm_run_static_scratch: one
 * 128 x 256 float32 partial tile for each of at most
 * SGEMM_STATIC_SCRATCH_MAX_CTAS CTAs (19,922,944 bytes), then one 32-bit
 * flag per CTA padded to 768 bytes: 19,923,712 bytes (19.0 MiB) in all,
 * reserved in device memory for each device whose context loads it.
 */
#define SGEMM_STATIC_SCRATCH_MAX_CTAS 152
#define SGEMM_STATIC_SCRATCH_BYTES ((size_t)SGEMM_STATIC_SCRATCH_MAX_CTAS * 128 * 256 * 4 + 768)

/*
 * C = alpha*A*B + beta*C with no plan and no memory allocation: the
 * 128 x 256 transposed-A kernel with its stream-K tail.  The pages have no
 * counterpart to this entry point.  They describe the kernels, not how a
 * library hands them workspace; it exists for deployment.
 *
 * Who cannot allocate, and why:
 *   - a caller inside a framework whose caching allocator already holds the
 *     device's memory (PyTorch's, for one).  cudaMalloc can then fail even
 *     though the framework has free blocks, and memory taken outside the
 *     pool is not given back to it.
 *   - a caller on a latency-bound path.  cudaFree waits for the whole
 *     device, and cudaMalloc can take far longer than a GEMM.
 *   - a caller with nowhere to keep a plan, such as a hook called per batch
 *     with no set-up or tear-down of its own.  Making and destroying a
 *     stream-K plan on every call would allocate and free each time.
 *
 * Arguments are sgemm_plan's dimensions and leading dimensions followed by
 * sgemm_run's arguments, with the same meaning, layout and ownership; A, B,
 * C are device pointers on the current device.  Enqueues on `stream` and
 * returns.  Results are bit-identical to sgemm_run of a plan made with the
 * variant "tmat_128x256x32_s3_b1" (k_order=split when the tail is split);
 * like plans, it honours the SGEMM_NO_STREAMK environment variable, which
 * turns the split off.
 *
 * Scratch: the stream-K workspace and its flags sit in one file-scope
 * __device__ array of SGEMM_STATIC_SCRATCH_BYTES (see above).  Only the
 * flags must start at zero: the first call on each device clears them,
 * and they are cleared again when the call counter wraps.  A partial tile
 * is always written before its flag is raised, so the workspace needs no
 * clearing.
 *
 * First-call set-up, once per device, with that device current:
 *   - looks up the array's device address (cudaGetSymbolAddress, which
 *     loads the module holding it);
 *   - sets the kernel's shared-memory limit and reads its occupancy;
 *   - clears the flags with cudaMemsetAsync on `stream`.
 * Make that first call before any stream capture.  After set-up a call
 * makes no allocation, host or device.
 *
 * Concurrency: every call on a device shares that device's scratch.  Calls
 * that overlap in time race and give wrong results or SGEMM_ERR_TIMEOUT in
 * the status word.  This holds for calls on two streams not ordered by
 * events, and for calls from two host threads at once.  Serialise them:
 * one stream, or event ordering.
 *
 * Errors:
 *   - SGEMM_ERR_INVALID_ARG and the dimension rules are as for sgemm_plan
 *     and sgemm_run.
 *   - SGEMM_ERR_UNSUPPORTED when this kernel cannot take the layout: lda or
 *     ldb not a multiple of 4, or A or B not 16-byte aligned.  These need
 *     sgemm_plan and sgemm_run.
 *   - SGEMM_ERR_UNSUPPORTED when C shares its address span with A or B
 *     (the conservative span test of sgemm_run): the kernel reads A and B
 *     while other CTAs write C.  A and B may alias each other.
 *   - SGEMM_ERR_UNSUPPORTED also when the call would need more scratch than
 *     the array holds: a stream-K grid of more than
 *     SGEMM_STATIC_SCRATCH_MAX_CTAS CTAs, on a device with more SMs than
 *     GB300's 152.  On GB300 every shape fits.
 * M == 0 or N == 0 launches nothing.  K == 0 or alpha == 0 scales C by
 * beta and uses no scratch.
 */
sgemm_status_t sgemm_run_static_scratch(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                        int64_t ldc, float alpha, const float *A, const float *B,
                                        float beta, float *C, void *stream);

/*
 * Measurement aid, not a product: the FP32 FMA pipe's achievable rate on
 * the current device.
 *   - Kernel: the FFMA kernels' accumulation pattern without their loads,
 *     run by two 256-thread CTAs per SM. paired = 1: FFMA2 on 4 x 8 pair
 *     accumulators (two A rows times one broadcast B value, the form the
 *     FFMA kernels issue). paired = 0: scalar FFMA on an 8 x 8 outer
 *     product. Either way each thread does 128 FLOP per step.
 *   - *tflops: the rate measured with CUDA events over one launch, after
 *     one warm-up launch.
 *   - *sm_mhz: the SM clock read inside the kernel, as cycles per
 *     nanosecond of the global timer between the start and end of its
 *     first CTA.
 *   - Behaviour: synchronous (about 1 ms on GB300) on a private stream.
 *     SGEMM_ERR_INVALID_ARG for NULL outputs or paired not 0 or 1.
 * The FFMA roofline's nominal denominator is SMs x 128 x 2 x clock; the
 * pages report an FMA-only test reaching 96% of that rate ("Writing a Fast
 * Matmul in CUDA, Step by Step", the measurement set-up). This gives the
 * same figure for GB300.
 */
sgemm_status_t sgemm_probe_ffma(int paired, double *tflops, double *sm_mhz);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_GB300_H */
