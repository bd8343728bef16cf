/*
 * pent.h — C ABI of the GB300 batched pentadiagonal solver library (libpent.so).
 *
 * The library solves many independent pentadiagonal systems A x = f at once,
 * the linear solve behind semi-implicit stepping of 1-D hyperdiffusion and
 * Cahn–Hilliard,  (I + sigma D4) C^{n+1} = RHS^n,  D4 = [1, -4, 6, -4, 1]/dx^4.
 * Source: "cuPentBatch – A batched pentadiagonal solver for NVIDIA GPUs"
 * (Gloster et al., arXiv 1807.07382).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Bands.  Row i (0-based) of a matrix holds a[i] at column i-2, b[i] at i-1,
 *   c[i] at i, d[i] at i+1, e[i] at i+2 — the naming of the page's
 *   factorisation steps (alpha_1 = c_1, beta_2 = b_2, delta_1 = e_1/alpha_1,
 *   eps_i = a_i).  Non-cyclic: entries whose column is outside 0..N-1 are
 *   ignored.  Cyclic (periodic, matrix (7c)): the column wraps modulo N.
 * Interleaved layout.  A batch of vectors is one array of N rows of `batch`
 *   elements; element i of system s lives at index i*batch + s (row i holds
 *   entry i of every system; the page's "interleaved data layout").
 * Memory.  Pointers named *_host are host memory; every other array pointer
 *   is device memory of the current CUDA device, owned by the caller, which
 *   must stay valid until the work queued on `stream` has finished.
 * Streams.  `stream` is a cudaStream_t passed as void*; NULL is the legacy
 *   default stream.  Solves are asynchronous (stream ordered).
 * Errors.  Every call returns a pent_status.  Argument errors are detected on
 *   the host before anything is queued, and nothing is modified.  A failed
 *   launch returns PENT_ERR_CUDA.  No entry point aborts, traps or prints.
 *   No entry point falls back to host computation: every solve runs in the
 *   library's CUDA kernels.
 */
#ifndef PENT_H
#define PENT_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PENT_OK = 0,
  PENT_ERR_INVALID_ARG = 1, /* bad size, null pointer, wrong plan kind         */
  PENT_ERR_ZERO_PIVOT = 2,  /* zero or non-finite pivot / singular 2x2 border  */
  PENT_ERR_CUDA = 3,        /* a CUDA call or kernel launch failed             */
  PENT_ERR_ALLOC = 4,       /* device or host allocation failed                */
  PENT_ERR_UNSUPPORTED = 5  /* valid request the library does not implement   */
} pent_status;

typedef enum { PENT_F64 = 0, PENT_F32 = 1 } pent_dtype;

/* Kernel variants of the shared-matrix solves (for tests and benchmarks;
 * PENT_VARIANT_AUTO picks one by shape). */
typedef enum {
  PENT_VARIANT_AUTO = 0,
  PENT_VARIANT_THREAD = 1,    /* one thread per system, native arithmetic of the plan dtype */
  PENT_VARIANT_THREAD_DF = 2, /* one thread per system, fp64 plans computed in double-float
                                 (pairs of fp32) on the FP32 pipe.  For shared-matrix
                                 plans this is the twisted kernel, which writes g over f
                                 as it sweeps and so cannot rescale a system: its pairs
                                 cover |values| in (2^-100, 2^127) only, and AUTO never
                                 picks it                                              */
  PENT_VARIANT_SPLIT = 3      /* each system split over a warp (partitioned solve)       */
} pent_variant;

typedef struct pent_plan_s* pent_plan;

/*
 * pent_factor — factor a shared matrix once (the page's factor/solve split,
 * "cuPentBatchConstant": factorisation steps 1–14 done once, reused by every
 * solve).  For cyclic = 1 it also precomputes the pieces of Navon's bordering
 * (eqs. (8)–(12)) that the page says to store once: E = leading (N-2)x(N-2)
 * block, the 2x2 inverse of B - H^T E^{-1} G and the vectors for H^T E^{-1}
 * and E^{-1} G.
 *   bands_host : HOST, 5*N doubles, row-major [5][N] = a, b, c, d, e.
 *   N          : rows; >= 1 (non-cyclic) or >= 5 (cyclic).
 *   batch      : number of systems the plan will usually be called with
 *                (>= 1); used to choose the kernel variant.
 *   cyclic     : 0 or 1.
 *   dtype      : PENT_F64 or PENT_F32 — element type of the solve arrays.
 *                The factorisation itself is always computed in fp64.
 *   out        : receives the plan (owned by the caller; free with pent_destroy).
 * The factorisation runs on the current device and the call waits for it.
 * Returns PENT_ERR_ZERO_PIVOT if a pivot alpha_i is zero or not finite, or
 * if the 2x2 border block is singular.  On error *out is set to NULL.
 */
pent_status pent_factor(const double* bands_host, int N, int batch, int cyclic, pent_dtype dtype,
                        pent_plan* out);

/*
 * pent_solve — shared-matrix batched solve in place: forward substitution
 * L g = f then back substitution R x = g (the page's steps for g and x), or
 * for a cyclic plan the bordered solve (eqs. (11)–(12)).
 *   rhs_inout : DEVICE, interleaved [N][batch] of the plan dtype; holds f on
 *               entry and x on return.  Base address 16-byte aligned.
 *   batch     : >= 1.
 * fp64 plans (AUTO variant) compute in double-float on the FP32 pipe and keep
 * the whole fp64 range: every system is scaled by the power of two that puts
 * its largest |f| in [1, 2) before it is converted, and systems whose largest
 * entry is zero, subnormal, non-finite or beyond the scaled kernels' window
 * are solved in native fp64.  Accuracy is relative to each system's largest
 * |x| (about 1e-13 against an fp64 solve).
 * Ordering: the plan holds device state that a solve uses while it runs (the
 * block queue of the persistent kernel, the chunk summaries of long systems),
 * so solves with one plan must be ordered (issued on one stream, or separated
 * by events); solves on different streams at once need one plan each.  The
 * state is back in its initial form when a solve completes, so a solve
 * captured in a CUDA graph can be replayed.
 */
pent_status pent_solve(pent_plan plan, void* rhs_inout, int batch, void* stream);

/*
 * pent_solve_host — pent_solve for right-hand sides held in HOST memory: the
 * call copies them to the device, solves and copies the solutions back, with
 * the transfers overlapped with the solves.  A library service around
 * pent_solve (the page solves device-resident batches).
 *   rhs_host : HOST, interleaved [N][batch] of the plan dtype (f in); pinned
 *              (page-locked) memory for the copies to run asynchronously.
 *   x_host   : HOST, same shape (x out); may equal rhs_host.
 *   chunks   : number of column blocks of systems the batch is cut into for the
 *              copy-in / solve / copy-out pipeline.  0 picks blocks whose rows
 *              are at least 128 KB (narrower 2-D copies run below the copy
 *              engines' rate on GB300), at most 8.  Each block is a multiple of
 *              64 systems except possibly the last.
 * The plan allocates, on first use, three device staging buffers of one block
 * each and three streams; they live until pent_destroy.  The call is ordered on
 * `stream` like pent_solve (it forks from and joins back into it) and returns
 * before the work completes; the host arrays must stay valid and unmodified until
 * the stream reaches this point.  Calls on one plan must be ordered (for example
 * issued on one stream): they share the staging buffers.
 * Errors: as pent_solve; PENT_ERR_ALLOC if the staging buffers cannot be made.
 */
pent_status pent_solve_host(pent_plan plan, const void* rhs_host, void* x_host, int batch, int chunks,
                            void* stream);

/*
 * pent_factor_solve — per-system matrices, factor + solve in one call
 * ("cuPentBatchRewrite": a new matrix every call).  Unlike the page, the
 * bands are left unchanged.  Row i of system s:
 *   a_i x_{i-2} + b_i x_{i-1} + c_i x_i + d_i x_{i+1} + e_i x_{i+2} = f_i
 * (entries that fall outside the matrix are ignored).
 *   a, b, c, d, e : DEVICE, interleaved [N][batch] each, dtype elements,
 *                   16-byte aligned; not modified.
 *   rhs_inout     : DEVICE, interleaved [N][batch], 16-byte aligned; f in, x out.
 *   N, batch      : >= 1.
 *   work          : DEVICE scratch, 256-byte aligned, contents undefined
 *                   afterwards, of at least pent_factor_solve_needs_work()
 *                   bytes; NULL (with work_bytes 0) when that is 0 (fp32
 *                   systems of up to 512 rows, which the partitioned kernel
 *                   keeps on chip).  The page's Rewrite scheme overwrites the
 *                   caller's bands with the factors; this library keeps them
 *                   and asks the caller for the factor storage instead, in
 *                   line with its rule that the caller owns every device
 *                   buffer of a call.
 *   info          : DEVICE int[batch] or NULL.  info[s] = 0 if system s was
 *                   factored, else the 1-based row of the first zero or
 *                   non-finite pivot the kernel's elimination met (its x is
 *                   then not meaningful; the row may differ between variants).
 * Non-cyclic only.  Equivalent to pent_factor_solve_ex with PENT_VARIANT_AUTO.
 */
pent_status pent_factor_solve(const void* a, const void* b, const void* c, const void* d,
                              const void* e, void* rhs_inout, int N, int batch, pent_dtype dtype,
                              void* work, size_t work_bytes, int* info, void* stream);

/*
 * pent_factor_solve_ex — pent_factor_solve with the kernel chosen by the caller.
 *   variant : PENT_VARIANT_THREAD — one thread per system (the page's Rewrite
 *             scheme): gamma_i and delta_i go to `work`, g_i over the
 *             right-hand side, read back by the backward sweep;
 *             PENT_VARIANT_SPLIT — fp32 and N <= 512 only: each system cut
 *             into chunks of 16 rows, one thread per chunk, its tile loaded
 *             into shared memory by TMA and kept on chip (partitioned
 *             elimination; the chunk-end pairs of unknowns by block parallel
 *             cyclic reduction), so memory sees the bands and f once and x
 *             once; `work` is not used and may be NULL;
 *             PENT_VARIANT_THREAD_DF — fp64 only: THREAD's sweeps in
 *             double-float (pairs of floats on the FP32 pipe, ~2^-47 relative),
 *             inputs and outputs fp64, the scratch holding pairs; every row is
 *             scaled by the power of two of its diagonal and the solution by a
 *             per-system power of two, and from the first row the pairs
 *             cannot represent (or a zero, subnormal or non-finite diagonal or
 *             right-hand side) the thread continues in native fp64, so the
 *             whole fp64 range is kept;
 *             PENT_VARIANT_AUTO — SPLIT where it applies, else THREAD_DF for
 *             fp64, else THREAD.
 *   block_size : 0 — a..e and rhs_inout interleaved [N][batch], element (i, s)
 *             at i * batch + s; bs > 0 — the block-interleaved layout of
 *             "Simulating the behavior of the human brain on GPUs", section
 *             4.1.1: blocks of bs systems, each block an interleaved [N][bs]
 *             array, (i, s) at (s / bs) * N * bs + i * bs + s % bs; batch must
 *             be a multiple of bs.  The SPLIT kernel loads a block-interleaved
 *             tile with one box per array when bs is a multiple of 16.  `work`
 *             keeps its own layout whatever bs is.
 *   other arguments as for pent_factor_solve; `work` is required (non-NULL,
 *   large enough, 256-byte aligned) only when THREAD runs.
 * Errors: PENT_ERR_INVALID_ARG for null or misaligned pointers, N or batch < 1,
 * a bad dtype, variant or block_size, or a missing or short work buffer where
 * THREAD or THREAD_DF runs; PENT_ERR_UNSUPPORTED for SPLIT outside fp32 /
 * N <= 512 and for THREAD_DF outside fp64.  Nothing is
 * queued on an error.
 */
pent_status pent_factor_solve_ex(const void* a, const void* b, const void* c, const void* d,
                                 const void* e, void* rhs_inout, int N, int batch, pent_dtype dtype,
                                 pent_variant variant, int block_size, void* work, size_t work_bytes,
                                 int* info, void* stream);

/* Bytes of device scratch the one-thread-per-system kernels of
 * pent_factor_solve_ex use for (N, batch, dtype) (variants THREAD and
 * THREAD_DF). */
size_t pent_factor_solve_work_bytes(int N, int batch, pent_dtype dtype);

/* Bytes of device scratch pent_factor_solve (the AUTO variant) needs for
 * (N, batch, dtype): 0 where it picks the partitioned kernel (fp32, N <= 512),
 * else pent_factor_solve_work_bytes(). */
size_t pent_factor_solve_needs_work(int N, int batch, pent_dtype dtype);

/*
 * pent_factor_solve_noalloc — pent_factor_solve for callers that cannot
 * allocate device memory.  The paper has no counterpart; this is a library
 * service.  Some callers cannot call cudaMalloc: an application that reserved
 * all device memory for its own pool at start-up and does not let libraries
 * allocate, or a time-critical loop where cudaMalloc/cudaFree are ruled out
 * because they may synchronise the device and take unbounded time.
 *
 * Same kernel and results as pent_factor_solve.  fp32 systems of up to 512
 * rows take the partitioned kernel, which needs no scratch; otherwise the
 * scratch for the factor coefficients is a fixed 16 MiB array inside the library (every GPU that
 * loads the library holds it until the process exits).  Nothing is allocated:
 * no cudaMalloc, cudaFree or allocating library routine is called.
 *   a..e, rhs_inout, N, batch, dtype, info : as for pent_factor_solve.
 * Limit, where the scratch is used (fp64, or N > 512): 2 * N * batch *
 * sizeof(element) must be <= 16 MiB (for example N = 300 with batch <= 3495
 * in fp64, or N = 1024 with batch <= 2048 in fp32); larger requests return
 * PENT_ERR_UNSUPPORTED and queue nothing.
 * Set-up: the first call on each device looks up the device address of the
 * array (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.
 * Sharing: every call uses the same array.  The kernel writes each scratch
 * entry before reading it, so nothing needs clearing between calls, but two
 * calls whose kernels overlap on the GPU (different streams, or different host
 * threads without ordering) race on the array; order them on one stream or
 * with events.
 */
pent_status pent_factor_solve_noalloc(const void* a, const void* b, const void* c, const void* d,
                                      const void* e, void* rhs_inout, int N, int batch,
                                      pent_dtype dtype, int* info, void* stream);

/*
 * hyperdiffusion_step — nsteps of C <- A^{-1} C with a cyclic plan, i.e. the
 * semi-implicit step (I + sigma D4) C^{n+1} = C^n of the hyperdiffusion
 * equation (eq. (4)) with periodic boundaries, the plan built from the bands
 * [sigma, -4 sigma, 1 + 6 sigma, -4 sigma, sigma].
 *   C_inout : DEVICE, interleaved [N][batch], plan dtype (must be PENT_F64).
 *   nsteps  : >= 0.
 */
pent_status hyperdiffusion_step(pent_plan plan, void* C_inout, int batch, int nsteps, void* stream);

/*
 * ch_step — nsteps of the semi-implicit Cahn–Hilliard scheme (eqs. (1a),
 * (2)) with mobility D = 1, periodic on N points:
 *   (I + gamma dt D4) C^{n+1} = C^n + dt D2[(C^n)^3 - C^n],
 * D2 = [1, -2, 1]/dx^2.  The plan must be cyclic, PENT_F64, built from the
 * bands of I + sigma D4 with sigma = gamma dt/dx^4.  The explicit right-hand
 * side is computed inside the solve kernel (no extra pass over memory).
 *   C_inout     : DEVICE, interleaved [N][batch] doubles.
 *   dt_over_dx2 : dt/dx^2 of the explicit D2 term.
 */
pent_status ch_step(pent_plan plan, void* C_inout, int batch, double dt_over_dx2, int nsteps,
                    void* stream);

/*
 * cn_step — nsteps of the Crank–Nicolson scheme for hyperdiffusion (eqs. (5)
 * and (6) of "cuPentBatch – A batched pentadiagonal solver for NVIDIA GPUs"),
 * periodic on N points:
 *   (I + sigma_x D4) C^{n+1} = (I - sigma_x D4) C^n,  sigma_x = dt / (2 dx^4).
 * The plan must be cyclic, PENT_F64, built from the bands of
 * A = I + sigma_x D4 ([sigma_x, -4 sigma_x, 1 + 6 sigma_x, -4 sigma_x, sigma_x]).
 * The explicit half is taken as 2I - A, so for any cyclic plan
 * A = I + (dt/2) L the call performs C <- A^{-1} (2I - A) C, the
 * Crank–Nicolson step of dC/dt = -L C.  Explicit half and solve run in one
 * kernel per step (no extra pass over memory).
 *   C_inout : DEVICE, interleaved [N][batch] doubles, 16-byte aligned.
 *   nsteps  : >= 0.
 * Errors: PENT_ERR_INVALID_ARG for a null or non-cyclic or fp32 plan, a null
 * or misaligned C_inout, batch < 1 or nsteps < 0 (nothing queued);
 * PENT_ERR_CUDA if a launch fails (steps already queued stay queued).
 */
pent_status cn_step(pent_plan plan, void* C_inout, int batch, int nsteps, void* stream);

/*
 * tri_factor_solve — batched tridiagonal systems with per-system matrices,
 * factor + solve in one call: the Thomas algorithm of "Simulating the
 * behavior of the human brain on GPUs" (Valero-Lara et al.), section 4.1,
 * in the interleaved one-thread-per-system layout of its section 4.1.1
 * (cuThomasBatch).  Row i of system s:
 *   a_i x_{i-1} + b_i x_i + c_i x_{i+1} = y_i   (a_0 and c_{N-1} are ignored).
 *   a, b, c   : DEVICE, dtype elements, layout given by block_size; not modified.
 *   rhs_inout : DEVICE, same layout; y in, x out.
 *   N, batch  : >= 1.
 *   block_size: 0 — interleaved [N][batch]: element (i, s) at i * batch + s.
 *               bs > 0 — the page's block-interleaved layout (section 4.1.1):
 *               blocks of bs systems, each block an interleaved [N][bs] array,
 *               blocks one after another: (i, s) at (s / bs) * N * bs + i * bs
 *               + s % bs.  batch must be a multiple of bs.  The SPLIT kernel
 *               loads a block-interleaved tile with one contiguous box per array
 *               when bs is a multiple of 16.
 *   variant   : PENT_VARIANT_THREAD — one thread per system, c'_i kept in `work`
 *               and y'_i written over the right-hand side (the page's scheme);
 *               PENT_VARIANT_SPLIT — fp32 and N <= 512 only: each system held
 *               in registers across a group of threads (chunks of 16 rows,
 *               partitioned elimination, chunk-end unknowns by parallel cyclic
 *               reduction), so memory sees a, b, c, y once and x once;
 *               PENT_VARIANT_THREAD_DF — fp64 only: THREAD's sweeps in
 *               double-float (pairs of floats on the FP32 pipe, ~2^-47
 *               relative), the scratch and y' holding pairs; rows scaled by
 *               their diagonal's power of two, the solution by a per-system
 *               power of two, native fp64 from the first row the pairs cannot
 *               represent: the whole fp64 range is kept;
 *               PENT_VARIANT_AUTO — SPLIT where it applies, else THREAD_DF for
 *               fp64, else THREAD.
 *   work      : DEVICE scratch of tri_factor_solve_work_bytes() bytes,
 *               256-byte aligned (may be NULL with work_bytes 0 when the SPLIT
 *               kernel runs); contents undefined afterwards.
 *   info      : DEVICE int[batch] or NULL.  info[s] = 0, or the 1-based row of a
 *               zero or non-finite pivot met by the kernel's elimination (the
 *               row may differ between variants); x of that system is then
 *               undefined.  No pivoting is done: use diagonally dominant or SPD
 *               matrices, as the page does.
 * Errors: PENT_ERR_INVALID_ARG for null or misaligned pointers, N or batch < 1,
 * a bad dtype, variant or block_size, or a short work buffer; PENT_ERR_UNSUPPORTED for
 * SPLIT outside fp32 / N <= 512 and for THREAD_DF outside fp64.  Nothing is queued on an error.
 */
size_t tri_factor_solve_work_bytes(int N, int batch, pent_dtype dtype);
pent_status tri_factor_solve(const void* a, const void* b, const void* c, void* rhs_inout, int N,
                             int batch, pent_dtype dtype, pent_variant variant, int block_size,
                             void* work, size_t work_bytes, int* info, void* stream);

/* Select the kernel variant of a plan (PENT_VARIANT_AUTO restores the default).
 * PENT_ERR_UNSUPPORTED if the variant does not exist for this plan.  The
 * twisted variant (PENT_VARIANT_THREAD_DF on a shared-matrix plan) has its own
 * tables, which the default path never uses: the first selection of it makes
 * them, synchronously, so do not select it while work on the plan is queued
 * (PENT_ERR_CUDA if that fails). */
pent_status pent_set_variant(pent_plan plan, pent_variant variant);

/* The variant the next call on this plan with `batch` systems would use. */
pent_variant pent_get_variant(pent_plan plan, int batch);

/*
 * pent_set_option — tuning and testing hooks of a plan.  The defaults are the
 * measured best; the other values exist so that tests can run the code paths
 * against one another (every setting computes the same solve to within the
 * library's tolerance).  Nothing here has a counterpart on the pages.  The
 * call may rewrite the plan's device tables synchronously: do not call it
 * while work that uses the plan is queued.
 *   PENT_OPT_FIXED_GRID            1 (default): partitioned fp64 solves use the
 *                                  fixed-grid kernel where the plan qualifies;
 *                                  0: the TwoSum double-float kernel.
 *   PENT_OPT_SERIAL_CHUNK_SCAN     1: exact serial chunk scan in the partitioned
 *                                  kernels; 0 (default): the plan's truncated
 *                                  parallel scan.  Plans of systems too long
 *                                  for one CTA: PENT_ERR_UNSUPPORTED.
 *   PENT_OPT_BORDER_ALL_CHUNKS     1: periodic border correction in every chunk;
 *                                  0 (default): only where it exceeds 2^-60.
 *   PENT_OPT_MULTI_STEP            1 (default): nsteps >= 2 in one launch where
 *                                  supported; 0: one launch per time step.
 *   PENT_OPT_CHEAP_TERMS           1 (default): the multi-step kernel adds
 *                                  correction terms below 2^-24 to the low word
 *                                  alone; 0: every term in double-float.
 *   PENT_OPT_CHUNK_DEDUP           1 (default): long systems read one copy of
 *                                  bitwise-equal chunk tables; 0: each its own.
 *   PENT_OPT_TWISTED_RING          cp.async ring depth of the twisted kernel:
 *                                  4, 6 (default), 8 or 12; 0: register ring.
 *   PENT_OPT_STEPS_SYSTEMS         systems per CTA of the multi-step kernel:
 *                                  0 (default: by shape), 8 or 16.
 *   PENT_OPT_TWISTED_SYSTEMS_PER_CTA    register-ring twisted kernel: 64, 128,
 *                                  160, 256 (default) or 320.
 *   PENT_OPT_TWISTED_SYSTEMS_PER_THREAD 1 or 2 (default).
 *   PENT_OPT_TWISTED_PREFETCH_ROWS 4 (default) or 8.
 *   PENT_OPT_PERSISTENT_CTAS       CTAs of the persistent double-float kernels;
 *                                  0 (default): as many as fit on every SM.
 * Errors: PENT_ERR_INVALID_ARG for a null plan, an unknown option or a value
 * outside its list; PENT_ERR_CUDA if updating the device tables fails.
 */
typedef enum {
  PENT_OPT_FIXED_GRID = 1,
  PENT_OPT_SERIAL_CHUNK_SCAN = 2,
  PENT_OPT_BORDER_ALL_CHUNKS = 3,
  PENT_OPT_MULTI_STEP = 4,
  PENT_OPT_CHEAP_TERMS = 5,
  PENT_OPT_CHUNK_DEDUP = 6,
  PENT_OPT_TWISTED_RING = 7,
  PENT_OPT_STEPS_SYSTEMS = 8,
  PENT_OPT_TWISTED_SYSTEMS_PER_CTA = 9,
  PENT_OPT_TWISTED_SYSTEMS_PER_THREAD = 10,
  PENT_OPT_TWISTED_PREFETCH_ROWS = 11,
  PENT_OPT_PERSISTENT_CTAS = 12
} pent_option;
pent_status pent_set_option(pent_plan plan, pent_option option, int value);

/*
 * pent_plan_error — whether a kernel of this plan gave up: PENT_ERR_CUDA if a
 * kernel stopped because a bulk copy into shared memory did not complete
 * within its time limit (2 s) or could not be issued safely, PENT_OK
 * otherwise.  Such a kernel leaves the systems it had not finished unchanged
 * or partly solved.  Reads a device word of the plan synchronously (ordered
 * after the work already queued on the legacy default stream).  Library
 * service; nothing on the pages corresponds to it.
 */
pent_status pent_plan_error(pent_plan plan);

/* Free a plan (NULL is allowed).  Waits for nothing: the caller must not free
 * a plan while work using it is still queued. */
void pent_destroy(pent_plan plan);

/* cudaStreamSynchronize(stream) and report any pending CUDA error. */
pent_status pent_sync(void* stream);

/* Static, human-readable name of a status code. */
const char* pent_status_string(pent_status status);

/* Number of kernel launches this library has queued since it was loaded. */
unsigned long long pent_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* PENT_H */
