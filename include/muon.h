/*
 * muon.h - C ABI of a single-GPU Muon optimizer step for GB300 (sm_103a).
 *
 * What one step computes, per weight matrix W (m x n, row-major fp32):
 *   M   <- mu*M + G                         ("Muon is Scalable for LLM Training" blog, eq. (1))
 *   U    = mu*M + G                         (same page, Nesterov-style input)
 *   X0   = O(U) / ||U||_F                   (same page, Background; orientation O: transpose
 *                                            when m > n, "Scaling Muon for Diffusion
 *                                            Transformers" sec. 3.1)
 *   X_J  = J quintic Newton-Schulz steps    (blog eq. (2), (a,b,c) = (3.4445,-4.7750,2.0315)),
 *          carried in the r x r Gram space  (DMuon, "Gram Newton-Schulz"; r = min(m,n))
 *   W   <- W - lr*(0.2*sqrt(max(m,n))*O^{-1}(X_J) + wd*W)          (blog eq. (4))
 * RowNorm mode replaces X_J by R_eps(O(U)), each oriented row divided by
 * max(||row||_2, eps) (DiT paper sec. 3.1), with the same update scale.
 *
 * Conventions for every entry point:
 *  - Matrices are dense, row-major, contiguous, in device memory of the current
 *    CUDA device; params and momentum are fp32 and updated in place; grads are
 *    the plan's grad dtype and only read.  The caller owns all of them.
 *  - Pointer arrays (params, grads, momentum) are HOST arrays of n device
 *    pointers, in the order of the shapes given to muon_plan_create.  They may
 *    change from call to call; the array itself is read before the call returns.
 *  - stream is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    All device work is enqueued on it (muon_step_host and the overlapped
 *    fused/batched products also use streams of the plan, joined back into it);
 *    no call synchronises the host except muon_plan_create and
 *    muon_plan_destroy (the whole device: they allocate and free the workspace),
 *    muon_sync, muon_plan_tune, the muon_debug_copy_* calls, and muon_step_host
 *    with pageable host memory.
 *  - A plan is not thread-safe: its calls share one workspace, pinned pointer
 *    table and event set, so calls on one plan must not overlap, and steps of one
 *    plan issued to different streams must be ordered by the caller.  Separate
 *    plans are independent.
 *  - Errors: every argument is validated on the host before anything is
 *    launched, and an invalid call returns MUON_ERR_INVALID_ARG (or
 *    MUON_ERR_UNSUPPORTED) with no buffer touched.  A failed launch returns
 *    MUON_ERR_CUDA.  A device-side bounded wait that expires (a tensor-core
 *    pipeline stall) is recorded in the plan's device status word and returned
 *    by the next muon_sync as MUON_ERR_TIMEOUT.  No C++ exception crosses this
 *    boundary.
 */
#ifndef MUON_GB300_H
#define MUON_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MUON_OK = 0,
    MUON_ERR_INVALID_ARG = 1,   /* bad shape, null pointer, overlap, hyperparameter out of range */
    MUON_ERR_UNSUPPORTED = 2,   /* dtype / size the library does not handle */
    MUON_ERR_OOM = 3,           /* workspace allocation failed */
    MUON_ERR_CUDA = 4,          /* a CUDA runtime or launch error */
    MUON_ERR_TIMEOUT = 5,       /* a device-side bounded wait expired */
    MUON_ERR_NONFINITE = 6      /* a non-finite input norm (opts.check_finite), reported by muon_sync */
} muon_status;

typedef enum { MUON_F32 = 0, MUON_BF16 = 1 } muon_dtype;
typedef enum { MUON_MODE_NS = 0, MUON_MODE_ROWNORM = 1 } muon_mode;

/* Shape of one matrix as stored: rows x cols, row-major. */
typedef struct { int64_t rows, cols; } muon_shape;

typedef struct {
    /* nonzero: NS steps also write the orthogonalised update O (fp32, stored
       layout m x n) into the workspace so muon_debug_copy_update can return it */
    int32_t keep_update;
    /* nonzero: each step records CUDA events around its stages (read with muon_stage_times) */
    int32_t timing;
    /* nonzero: run every tensor-core product on the one-SM kernel (128 x 256 tiles)
       instead of the CTA-pair kernel (256 x 256 tiles, tcgen05 cta_group::2) */
    int32_t single_sm_gemm;
    /* nonzero: matrices with min(m, n) <= 128 also take the batched products instead of
       the fused kernel that runs the whole step of such a matrix on one SM */
    int32_t generic_small;
    /* plans holding both fused (min(m, n) <= 128) and batched matrices run the
       two concurrently: the fused kernel on all SMs but 2 x chain_clusters, the
       batched products on a second stream forked from and joined back into the
       caller's stream with events.  0: chosen from the plan's work estimate
       (overlap only when the fused matrices hold most of the work); > 0: that
       many CTA pairs for the batched products; < 0: no overlap (the fused
       kernel, then the batched products, on the caller's stream).  Results do
       not depend on this choice. */
    int32_t chain_clusters;
    /* > 0: the plan accepts muon_step_ex calls with up to max_ns_steps Newton-Schulz
       steps (at most 100) and restart periods below ns_steps.  It reserves a second
       X buffer per matrix and runs every matrix on the batched path.  0: ns_steps
       <= 5 in one segment, matrices with min(m, n) <= 128 on the fused kernel. */
    int32_t max_ns_steps;
    /* > 0: cap on the plan's device workspace in bytes.  The NS step then runs in
       chunks of matrices (momentum, SYRK, recursion, final product + update per
       chunk) whose X0 and r x r buffers share one region; results are the same.
       muon_plan_create returns MUON_ERR_OOM if the cap cannot hold the per-matrix
       tables plus the buffers of the largest single matrix.  0: no cap (one chunk).
       Negative: MUON_ERR_INVALID_ARG. */
    int64_t workspace_bytes;
    /* > 1: split the matrices into about this many chunks (the region each chunk
       needs is at most 1/chunks of the whole, and at least one matrix's), so that
       muon_step_host can overlap one chunk's host copies with another chunk's
       compute.  Results are the same.  0 or 1: chunks only as workspace_bytes
       requires.  Negative: MUON_ERR_INVALID_ARG. */
    int32_t chunks;
    /* nonzero: symmetric r x r results (G, P, T, Q) stored whole on every launch.  0:
       chunks whose batched matrices have r and c multiples of 64 store them as their
       lower triangle (256 x 256 tiles at or below the diagonal; the products read the
       blocks above it from the mirror position), which saves the mirrored half of the
       epilogue's stores.  Results are the same. */
    int32_t full_symmetric;
    /* Which matrices with min(m, n) <= 128 run the NS step in fp32 on CUDA cores (one
       matrix per CTA, the Gram recursion of DMuon's "Gram Newton-Schulz" with every
       product in fp32) instead of on the tensor cores.  A nearly square Gaussian
       matrix has singular values near zero, which the quintic amplifies by about
       a^5 ~ 485; the tensor-core recipe (bf16 X0 and Q, fp16 Gram recursion) moves
       its O by 1.3e-2 to 8e-2, the fp32 path by about 1e-5.  0: matrices with
       max(m, n) < 1.25 min(m, n); > 0: every matrix with min(m, n) <= 128 (slower for
       long matrices: the fp32 products run at CUDA-core rate); < 0: none.  Plans with
       max_ns_steps > 0 never use it.  generic_small does not apply to these matrices. */
    int32_t small_fp32;
    /* nonzero: every step also checks its inputs for NaN and infinity: the squared norm
       of each matrix's Nesterov input U (NS steps) and of each RowNorm row (RowNorm
       steps) must be finite.  A non-finite one is recorded in the plan's device status
       word and the next muon_sync returns MUON_ERR_NONFINITE.  The step still runs (the
       update of such a matrix is then not finite).  0: no check. */
    int32_t check_finite;
    /* Precision of the batched products (matrices on neither one-CTA kernel).  Level 1
       carries every r x r buffer (G, P, T, Q) as two fp16 parts and the final Q as
       two bf16 parts (value = hi + lo, about 21 and 16 significant bits), each product
       running as K-concatenated passes over the parts (3 for two split operands);
       level 2 also splits X0 into two bf16 parts (the SYRK and the final product read
       both).  Level 1 triples the r x r products' tensor work, level 2 also the SYRK
       and the final product.  Symmetric results of split buckets are stored whole.
       0: level 1 for nearly square buckets (max(m, n) < 1.25 min(m, n)) with
       min(m, n) <= split_max_r, whose O the plain recipe moves by 1e-2 to 2.5e-2;
       1 or 2: that level for every batched bucket; < 0: never. */
    int32_t precision;
    /* Largest min(m, n) that precision 0 splits (0: 1024). */
    int32_t split_max_r;
    /* NULL, or a host array of n row counts (read during muon_plan_create only) that
       makes the plan a RowNorm plan over dim-0 shards: matrix i is a block of rows of a
       full matrix of full_rows[i] >= rows rows and the same columns ("Scaling Muon for
       Diffusion Transformers" sec. 1 and 2.3: RowNorm steps on dim-0-sharded momentum).
       Orientation and the update scale follow the full shape: when full_rows[i] > cols
       the RowNorm rows are stored columns spanning every shard, and their squared norms
       are summed across shards between muon_rownorm_shard_stats and
       muon_rownorm_shard_apply; otherwise each stored row is complete in the shard.
       Such a plan runs only those two calls (the others return MUON_ERR_UNSUPPORTED). */
    const int64_t* full_rows;
    /* NULL, or a host array of n entries (read during muon_plan_create only) choosing the
       precision of each matrix on the batched products: < 0 plain, 1 or 2 that split level,
       0 the plan-wide rule of opts.precision.  Matrices of one oriented shape with different
       entries form separate buckets.  Matrices on the one-CTA kernels ignore it.  A caller
       (or MuonPlan.select_precision in the Python binding) can thus keep the plain recipe
       where it meets a tolerance on its own data and split only where it does not. */
    const int32_t* precision_of;
} muon_plan_opts;

typedef struct muon_plan_s* muon_plan;

/*
 * muon_plan_create - plan a step for a fixed list of matrix shapes ("muon_plan(shapes)").
 *   shapes     host array of n shapes: 1 <= rows, cols <= 2^20 and
 *              min(rows, cols) <= 32768, else MUON_ERR_UNSUPPORTED.
 *   grad_dtype dtype of every gradient: MUON_F32 or MUON_BF16.
 *   opts       may be NULL (all zero).
 *   out        receives the plan.
 * Orients every shape to r x c (r = min, c = max; DiT paper sec. 3.1),
 * buckets equal (r, c) so each Gram Newton-Schulz product runs as one grouped
 * launch over all matrices of all buckets (DMuon, batching same-shape matrices),
 * and allocates the workspace once (bf16 X0, the fp16 r x r Gram-space buffers
 * and a bf16 copy of Q, per-matrix tables, launch lists, status word) on the
 * current device.  The plan owns the workspace; muon_plan_destroy frees it.
 * Returns MUON_ERR_OOM if cudaMalloc (or a host allocation) fails.
 */
muon_status muon_plan_create(const muon_shape* shapes, int32_t n, muon_dtype grad_dtype,
                             const muon_plan_opts* opts, muon_plan* out);

/*
 * muon_plan_workspace_size - size the plan muon_plan_create would build for the
 * same shapes, grad_dtype and opts, on the host alone: no CUDA call is made, so
 * it works without a GPU.
 *   bytes      receives the device workspace muon_plan_create would allocate (its
 *              one cudaMalloc; muon_plan_info reports the same figure).
 *   n_buckets  receives the number of (r, c) buckets, counted per chunk.
 *   n_chunks   receives the number of chunks the NS step would run in.
 * Any output pointer may be NULL.  Same argument checks and codes as
 * muon_plan_create, including MUON_ERR_OOM when opts->workspace_bytes cannot
 * hold the per-matrix tables plus the buffers of the largest single matrix.
 */
muon_status muon_plan_workspace_size(const muon_shape* shapes, int32_t n, muon_dtype grad_dtype,
                                     const muon_plan_opts* opts, int64_t* bytes, int32_t* n_buckets,
                                     int32_t* n_chunks);

/*
 * muon_partition - owner assignment of matrices to `world` GPUs (DMuon technical
 * summary sec. 2: every matrix has exactly one owner rank, which keeps its momentum
 * and runs its Newton-Schulz step once; the other ranks receive the updated
 * parameters).  Host only, no CUDA call; deterministic, so every rank computes the
 * same assignment from the same arguments without communicating.
 *   shapes, n  the matrices, as for muon_plan_create (same limits).
 *   world      number of ranks, 1 .. 65536.
 *   cost       NULL, or n non-negative finite costs (for example measured seconds per
 *              matrix).  NULL: a model of one GB300 step, per matrix the larger of
 *              its tensor work ((3 r^2 c + 17 r^3) FLOPs at 1.5e15 FLOP/s, symmetric
 *              products counted at half; none for min(m, n) <= 128) and its memory
 *              traffic (24 bytes per element at 6.8e12 B/s), where r = min(m, n) and
 *              c = max(m, n).
 *   owner      receives n ranks in [0, world).
 *   load       NULL, or receives `world` summed costs.
 * The assignment is longest-processing-time first (DMuon's greedy fallback to its
 * MILP): matrices in decreasing cost (ties by index) each go to the rank with the
 * least load so far (ties by rank).  MUON_ERR_INVALID_ARG on a bad argument.
 */
muon_status muon_partition(const muon_shape* shapes, int32_t n, int32_t world, const double* cost, int32_t* owner,
                           double* load);

/*
 * muon_plan_destroy - wait for the device to go idle (cudaDeviceSynchronize, so
 * no step of the plan is still running), then free everything the plan owns: its
 * workspace, streams, events and pinned pointer table.  NULL is ignored.  The
 * handle must not be used afterwards.
 */
void muon_plan_destroy(muon_plan p);

/*
 * muon_step - one Muon step over every matrix of the plan.
 *   params, grads, momentum  host arrays of n device pointers (see conventions).
 *   lr >= 0, wd >= 0, 0 <= mu < 1, all finite.
 *   ns_steps in [0, 5]: Newton-Schulz iterations (5 in the pages; 0 gives O = X0).  The
 *     Gram-space recursion carries G in fp16; a rounding-level negative eigenvalue of G
 *     grows about 12x per step, so beyond five steps it can diverge on rank-deficient or
 *     large square inputs.  Larger values return MUON_ERR_INVALID_ARG.
 *   mode MUON_MODE_NS, or MUON_MODE_ROWNORM (then equal to muon_rownorm_step with eps = 1e-8).
 * A matrix whose Nesterov input U is all zero gets O = 0 (only weight decay acts).
 * params and momentum must not overlap each other, the grads, or any other matrix.
 */
muon_status muon_step(muon_plan p, float* const* params, const void* const* grads,
                      float* const* momentum, float lr, float wd, float mu,
                      int32_t ns_steps, muon_mode mode, void* stream);

/*
 * muon_step_ex - muon_step in NS mode with the Newton-Schulz coefficients and
 * the evaluation schedule as arguments.
 *   coeffs: (a, b, c) of the step X <- aX + b(XX^T)X + c(XX^T)^2 X (blog eq. (2));
 *     NULL: the pages' (3.4445, -4.7750, 2.0315).  Cubic NS is (1.5, -0.5, 0).
 *   restart: the Gram recursion (DMuon, "Gram Newton-Schulz") runs in segments of
 *     at most `restart` steps (1..5; 0: 5).  After every segment but the last the
 *     iterate X <- Q X is formed explicitly (bf16) and the next segment's Gram
 *     matrix is computed from it: the same iteration in exact arithmetic, with the
 *     fp16 recursion restarted before rounding errors in near-null directions of G
 *     can grow.  restart = 1 is the direct form of eq. (2).
 *   ns_steps: 0 .. 5, or up to opts.max_ns_steps on plans created with it.
 * Runs with more than one segment need a plan created with opts.max_ns_steps > 0
 * (MUON_ERR_UNSUPPORTED otherwise).  Other arguments and errors as muon_step.
 */
muon_status muon_step_ex(muon_plan p, float* const* params, const void* const* grads, float* const* momentum,
                         float lr, float wd, float mu, int32_t ns_steps, const float* coeffs, int32_t restart,
                         void* stream);

/*
 * muon_step_host - muon_step for gradients that arrive from host memory and
 * parameters that go back to it, with the copies overlapped with the compute.
 *   grads_host   host array of n pointers to the gradients in host memory (grad
 *                dtype, stored shape).  Pinned memory lets the copies run
 *                asynchronously; with pageable memory each copy blocks the caller.
 *   grads        host array of n device pointers the gradients are copied to
 *                (caller-owned, as in muon_step); the step reads them there.
 *   params_host  NULL (no copy back), or a host array of n pointers to host
 *                buffers (fp32, stored shape) that receive the updated parameters.
 *   params, momentum, lr, wd, mu, ns_steps, mode: as muon_step (RowNorm with eps 1e-8).
 * NS mode runs chunk by chunk (opts.chunks, opts.workspace_bytes): one copy
 * stream of the plan copies the gradients in chunk order, each chunk's momentum
 * kernel waits only for its own chunk's gradients, and a second copy stream
 * copies each chunk's parameters back as soon as that chunk's final product has
 * run, while the next chunks compute.  RowNorm mode runs chunk by chunk in the
 * same way (eps = 1e-8).  The copies in are ordered after the work already on
 * `stream` (which may still read the previous gradients), and `stream` waits for
 * the last copy back: once `stream` is synchronised, params_host holds the
 * result.  Errors as muon_step; a null grads_host (or null entry of either host
 * array) is MUON_ERR_INVALID_ARG, checked before anything is enqueued.
 */
muon_status muon_step_host(muon_plan p, float* const* params, const void* const* grads, float* const* momentum,
                           const void* const* grads_host, float* const* params_host, float lr, float wd,
                           float mu, int32_t ns_steps, muon_mode mode, void* stream);

/*
 * muon_rownorm_step - one RowNorm step (DiT paper sec. 3, "periodic RowNorm Muon"):
 *   M <- mu*M + G;  U = mu*M + G;  R = R_eps(O(U)) over the rows of the oriented
 *   matrix (stored columns when m > n);  W <- W - lr*(0.2*sqrt(max(m,n))*R + wd*W).
 *   eps > 0 and finite.  Other arguments as muon_step.
 */
muon_status muon_rownorm_step(muon_plan p, float* const* params, const void* const* grads,
                              float* const* momentum, float lr, float wd, float mu,
                              float eps, void* stream);

/*
 * muon_rownorm_shard_stats / muon_rownorm_shard_apply - one RowNorm step of a plan
 * created with opts.full_rows (dim-0 shards; "Scaling Muon for Diffusion Transformers"
 * sec. 1 and 2.3: on RowNorm steps only the norm statistics of rows that span ranks are
 * all-reduced).
 *   stats: M <- mu M + G for every matrix; matrices whose RowNorm rows are complete in
 *     the shard (full_rows <= cols) are also normalised and applied (W updated); for the
 *     others, writes this shard's per-column sums of U^2 (U = mu M + G) into colsq.
 *   colsq: device buffer of muon_plan_info's colsq_len floats, caller-owned; matrix by
 *     matrix in plan order, each padded to a multiple of 4 floats (padding written as 0).
 *     Between the two calls the caller sums colsq element-wise over all shards of the
 *     same matrices (for example an all-reduce across ranks, in place).
 *   apply: W <- W - lr (0.2 sqrt(max(full_rows, cols)) U / max(sqrt(colsq), eps) + wd W)
 *     for the spanning matrices, with U recomputed from G and the new M.  params, grads
 *     and momentum must be those of the stats call, unchanged in between.
 * Arguments and errors as muon_rownorm_step; MUON_ERR_UNSUPPORTED on a plan without
 * opts.full_rows.  With opts.check_finite, apply checks the summed squared norms.
 */
muon_status muon_rownorm_shard_stats(muon_plan p, float* const* params, const void* const* grads,
                                     float* const* momentum, float lr, float wd, float mu, float eps, float* colsq,
                                     void* stream);
muon_status muon_rownorm_shard_apply(muon_plan p, float* const* params, const void* const* grads,
                                     float* const* momentum, float lr, float wd, float mu, float eps,
                                     const float* colsq, void* stream);

/*
 * muon_plan_tune - a profiled planner (DMuon's per-shape autotuning, on one GPU): times
 * the plan's launch choices that change only speed on the caller's buffers and keeps
 * the fastest.  Candidates: for chunks holding both fused (min(m, n) <= 128) and
 * batched matrices, the CTA pairs the batched products get beside the fused kernel
 * (none, the work estimate's choice, half and one and a half times it; only when
 * opts.chain_clusters is 0), and symmetric results stored as the lower triangle or
 * whole (chunks where opts.full_symmetric leaves the choice).
 * Every candidate gives bitwise the same results.  Each candidate runs one warm-up
 * and `reps` timed NS steps (ns_steps 5): params and momentum are updated as by that
 * many ordinary steps, so tune on scratch copies or count the calls as training
 * steps.  reps in [1, 100]; *ms_out (may be NULL) receives the chosen candidate's ms
 * per step.  Synchronises stream; errors as muon_step (MUON_ERR_INVALID_ARG for reps).
 */
muon_status muon_plan_tune(muon_plan p, float* const* params, const void* const* grads, float* const* momentum,
                           float lr, float wd, float mu, int32_t reps, float* ms_out, void* stream);

/*
 * muon_sync - wait for the plan's work on stream, then read and clear the
 * device status word.  Returns MUON_ERR_TIMEOUT if a bounded device wait
 * expired since the last muon_sync, else MUON_ERR_NONFINITE if a step of a plan
 * created with opts.check_finite met a non-finite input norm since then,
 * MUON_ERR_CUDA on a CUDA error.
 */
muon_status muon_sync(muon_plan p, void* stream);

/*
 * muon_debug_wait_timeout - test hook for the bounded device waits: enqueues on
 * stream one mbarrier wait whose phase nothing completes, bounded at limit_us
 * microseconds (1 .. 1e6).  The wait gives up, records the timeout in the plan's
 * status word and the kernel returns, as every tensor-core kernel does when a
 * TMA load or MMA commit never arrives; the next muon_sync returns
 * MUON_ERR_TIMEOUT (and clears the word) and the plan stays usable.
 */
muon_status muon_debug_wait_timeout(muon_plan p, int32_t limit_us, void* stream);

/*
 * muon_debug_copy_update - copy the orthogonalised update O of matrix i from
 * the last NS step (stored layout, m x n fp32) into dst (device memory, m*n
 * floats).  Needs opts.keep_update; synchronises stream.
 */
muon_status muon_debug_copy_update(muon_plan p, int32_t i, float* dst, void* stream);

/*
 * muon_debug_update_error - relative Frobenius difference ||O_i - ref|| / ||ref|| (the
 * plain norm of O_i when ref is zero) between the orthogonalised update O of matrix i from
 * the last NS step and ref (device memory, fp32, stored layout m x n), computed on the
 * device in fp64.  Needs opts.keep_update; synchronises stream.  Used to check one
 * precision of the Newton-Schulz recursion against another on the caller's own data.
 */
muon_status muon_debug_update_error(muon_plan p, int32_t i, const float* ref, double* rel, void* stream);

/*
 * muon_debug_copy_workspace - copy one workspace buffer of matrix i, as it is
 * after the last step, into dst (host or device memory), for step-by-step
 * parity checks.  Synchronises stream.  which:
 *   0 X0 workspace: bf16 U in the oriented layout, r rows of ld elements (unnormalised)
 *   1 G buffer 0, 2 G buffer 1: fp16 s*G with s = 2^round(log2 r), r rows of ld
 *   3 P, 4 T, 5 Q buffer 0, 6 Q buffer 1: fp16, r rows of ld
 *   7 bf16 Q of the final product: r rows of ld
 *   8 1/||U||_F: one fp32
 * *ld receives the leading dimension (elements) of the copied rows; the copy
 * is r*ld elements of 2 bytes (one 4-byte float for which = 8).
 * After a step with ns_steps = J, G buffer 0 holds s*G_0 when J <= 2, G
 * buffer 1 holds s*G_1 when J >= 2, buffer 3 holds P_J and buffer 7 holds Q_J.
 * Matrices with min(m, n) <= 128 on the fused kernel have no r x r buffers
 * (which 1-7 return MUON_ERR_UNSUPPORTED).  With a workspace cap the chunks
 * share these buffers: they hold the last chunk's matrices.
 */
muon_status muon_debug_copy_workspace(muon_plan p, int32_t i, int32_t which, void* dst, int32_t* ld,
                                      void* stream);

/*
 * muon_rownorm_matrix_noalloc - the RowNorm step of muon_rownorm_step for ONE
 * matrix, without allocating any device memory.  The pages have no
 * counterpart: this exists for callers that may not call cudaMalloc or have a
 * library call it - frameworks whose own pooling allocator owns all device
 * memory, processes under a hard memory budget, and latency-critical loops
 * that cannot afford cudaMalloc/cudaFree's implicit device synchronisation.
 *   param, momentum  fp32 rows x cols, updated in place; grad (grad_dtype) read.
 *   lr, wd, mu, eps  as muon_rownorm_step.
 * Scratch: when rows > cols the column statistics live in a 4 MiB array that is
 * part of the library image (every GPU that loads the library holds it until
 * the process exits); ceil(rows/64)*cols + cols floats must fit in 2^20, else
 * MUON_ERR_UNSUPPORTED is returned and nothing is launched.  Every call looks
 * the array's device address up in the current context (a host-side query with
 * no allocation and no synchronisation, so a context that was reset gets the
 * new address); the first call on a device may load the library's device code,
 * so make it before any stream capture.  A failed lookup or launch returns
 * MUON_ERR_CUDA and is reported by muon_last_error_detail.  Calls share the array, so calls that overlap
 * on the GPU (other streams, other host threads) race.  Nothing in the array
 * needs clearing: each call writes every word it reads.
 */
muon_status muon_rownorm_matrix_noalloc(float* param, const void* grad, float* momentum, int64_t rows,
                                        int64_t cols, muon_dtype grad_dtype, float lr, float wd, float mu,
                                        float eps, void* stream);

/* Human-readable name of a status code (static string). */
const char* muon_status_string(muon_status s);

/* Text of the last CUDA error this thread's calls turned into MUON_ERR_CUDA (static string). */
const char* muon_last_error_detail(void);

/* Plan introspection. */
typedef struct {
    int32_t n_matrices;
    int32_t n_buckets;
    int64_t workspace_bytes;
    int32_t launches_last_step;   /* kernels the last step enqueued */
    int32_t sm_count;
    int32_t n_chunks;             /* chunks the NS step runs in (opts.chunks, opts.workspace_bytes) */
    int32_t lower_chunks;         /* chunks storing symmetric results as the lower triangle */
    int32_t tuned_candidates;     /* launch choices muon_plan_tune measured (0: never tuned) */
    int32_t chain_clusters;       /* CTA pairs the batched products get beside the fused kernel (0: none) */
    int32_t split_buckets;        /* batched buckets in split precision (opts.precision) */
    int32_t fp32_buckets;         /* buckets on the fp32 kernel (opts.small_fp32) */
    int64_t colsq_len;            /* floats of the colsq buffer of the shard calls (0 without opts.full_rows) */
} muon_plan_info_t;

muon_status muon_plan_info(muon_plan p, muon_plan_info_t* info);

/*
 * muon_stage_times - device time (ms) per stage, summed over the steps run
 * since the previous call, measured with CUDA events recorded on each step's
 * stream (needs opts.timing; waits for those steps, then resets the sums).
 * Stages: [0] momentum + Nesterov + norm, [1] Gram SYRK, [2] r x r
 * Newton-Schulz products, [3] final product + fused apply, [4] RowNorm steps,
 * [5] the whole fused step of the matrices with min(m, n) <= 128 (one kernel).
 * n_stages <= 6.  flops (nullable, 3 entries) receives the algorithmic tensor
 * FLOPs of stages 1-3 over the same steps (symmetric products counted at half;
 * the fused matrices of stage 5 are not included).
 * Returns MUON_ERR_INVALID_ARG when no timed step was run.
 */
muon_status muon_stage_times(muon_plan p, float* ms, double* flops, int32_t n_stages);

#ifdef __cplusplus
}
#endif

#endif /* MUON_GB300_H */
