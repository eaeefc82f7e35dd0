/*
 * addln.h - C ABI of the GB300 (sm_103a) fused residual-Add + LayerNorm library.
 *
 * The operation, per row i of the row-major [rows, H] inputs X and R:
 *     A_i    = X_i + R_i                         residual add; A never goes to memory
 *                                                 unless the caller asks for it
 *     mean_i = (1/H) sum_j A_ij
 *     var_i  = (1/H) sum_j (A_ij - mean_i)^2     biased variance
 *     rstd_i = 1 / sqrt(var_i + eps)
 *     Y_ij   = gamma_j * (A_ij - mean_i) * rstd_i + beta_j
 * Sources: the residual-Add + LayerNorm subgraph and its fused traffic (read X
 * and R once, write Y once) are from "算子融合的收益量化" (fusion gains
 * quantified), section 1; the LayerNorm definition (two-pass mean/variance,
 * biased variance, eps inside the square root, per-element gamma and beta) is
 * fused_layernorm in "算子融合与Kernel合并" (operator fusion and kernel
 * merging), section 4.2; the optional extra outputs are that page's
 * multi-output pattern (section 4.4 table).
 *
 * Conventions shared by every entry point:
 *  - Pointers to tensors are caller-owned DEVICE pointers (cudaMalloc or any
 *    allocator, e.g. PyTorch's).  The library never allocates, frees or
 *    synchronises inside the compute calls; it only enqueues kernels.  The
 *    one exception is add_layernorm_fwd_host, which takes HOST pointers and
 *    also queues copies (its own entry below says how).
 *  - Layout: X, R, Y, A are contiguous row-major [rows, H] (row stride H) in
 *    the I/O dtype; gamma, beta are fp32 [H]; mean, rstd are fp32 [rows].
 *  - dtype: ADDLN_FP32, ADDLN_FP16 or ADDLN_BF16 (IEEE binary32, binary16,
 *    bfloat16).  Arithmetic is fp32 in registers; Y and A are rounded to the
 *    I/O dtype to nearest-even.
 *  - stream: a cudaStream_t passed as void*; NULL is the legacy default
 *    stream.  Work is asynchronous: a zero return means the arguments were
 *    valid and the launch was accepted, not that the kernel finished.
 *  - Misaligned pointers or an H that is not a whole number of 16-byte
 *    vectors are accepted; they select a slower element-wise path.
 *  - Aliasing: an output may be exactly the same buffer as X or R (same base
 *    pointer, in-place); every row is read in full before any of its outputs
 *    is written.  Any other overlap between an output and any input or other
 *    output returns ADDLN_ERR_ALIAS.
 *  - Errors are negative return codes; nothing aborts or exits.  All argument
 *    checks run before the first CUDA call, so a rejected call touches no
 *    device state.
 *  - rows == 0 is a successful no-op once dtype, H and eps are valid.
 *  - Thread safety: every entry point may be called from several host threads
 *    at once; addln_set_force_path and addln_set_wait_limit_ns change
 *    process-wide test settings.
 */
#ifndef ADDLN_H
#define ADDLN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* dtype codes */
#define ADDLN_FP32 0
#define ADDLN_FP16 1
#define ADDLN_BF16 2

/* return codes */
#define ADDLN_OK 0
#define ADDLN_ERR_NULL (-1)           /* a required pointer is NULL */
#define ADDLN_ERR_SHAPE (-2)          /* rows < 0, n < 0, H <= 0 or H > addln_max_hidden(dtype) */
#define ADDLN_ERR_DTYPE (-3)          /* unknown dtype code */
#define ADDLN_ERR_EPS (-4)            /* eps negative, NaN or infinite */
#define ADDLN_ERR_ALIAS (-5)          /* an output partially overlaps an input or another output */
#define ADDLN_ERR_LAUNCH (-6)         /* the CUDA launch failed (cudaGetLastError) */
#define ADDLN_ERR_UNSUPPORTED (-7)    /* a forced kernel path cannot run these arguments */
#define ADDLN_ERR_DEVICE_TIMEOUT (-8) /* a kernel's bounded wait on its own copy ran out */
#define ADDLN_ERR_CUDA (-9)           /* a CUDA runtime call outside a launch failed */
#define ADDLN_ERR_WORKSPACE (-10)     /* workspace missing, too small or not 16-byte aligned */
#define ADDLN_ERR_BOUNDS (-11)        /* checked build: a kernel skipped an out-of-bounds access */

/* kernel paths for addln_set_force_path */
#define ADDLN_PATH_AUTO 0
#define ADDLN_PATH_WARP_VEC 1   /* one warp per row, 16-byte vector loads, H <= 1024 */
#define ADDLN_PATH_CTA_TMA 2    /* one CTA per row, rows staged by TMA bulk copies */
#define ADDLN_PATH_CTA_VEC 3    /* one CTA per row, 16-byte vector loads */
#define ADDLN_PATH_SCALAR 4     /* element-wise loads; any alignment and H */

/*
 * Fused residual-Add + LayerNorm forward (definition above).
 *   x, r        [rows, H] inputs in dtype (required)
 *   gamma, beta [H] fp32 (required)
 *   y           [rows, H] output in dtype (required)
 *   resid_out   [rows, H] output A = X + R rounded to dtype, or NULL
 *   mean, rstd  [rows] fp32 outputs, each independently NULL-able
 *   eps         >= 0, added to the variance inside the square root.  eps = 0
 *               is accepted; a row of zero variance (all sums equal) then has
 *               rstd = +inf and Y = NaN, the 0/0 the definition gives there
 *               (mean is still the row's value)
 * Statistics use the unrounded fp32 sum, not A rounded to dtype.
 * Returns ADDLN_OK or a negative code.
 */
int add_layernorm_fwd(const void *x, const void *r, const float *gamma, const float *beta,
                      void *y, void *resid_out, float *mean, float *rstd,
                      int64_t rows, int64_t H, float eps, int dtype, void *stream);

/*
 * add_layernorm_fwd from HOST buffers to HOST buffers, the host-device
 * copies inside the call (the pages' operation, end to end; the pages have
 * no host-side entry point of their own).
 *   x_host, r_host        [rows, H] inputs in dtype, host memory (required)
 *   gamma_host, beta_host [H] fp32, host memory (required)
 *   y_host                [rows, H] output in dtype, host memory (required)
 *   resid_out_host        [rows, H] A = X + R rounded to dtype, or NULL
 *   mean_host, rstd_host  [rows] fp32, each independently NULL-able
 *   workspace             device memory of at least
 *                         add_layernorm_fwd_host_workspace_size(rows, H,
 *                         dtype, resid_out_host != NULL, mean_host || rstd_host)
 *                         bytes, 256-byte aligned; owned by the caller, not
 *                         touched by any other call while this one runs
 *   stream                the caller's stream; the kernels run on it, and it
 *                         waits for the last copy back, so synchronising it
 *                         completes the call
 * Two ways, chosen per call (add_layernorm_fwd_host_last_mode reports which):
 *   mapped   when the device can reach host memory (the pageable memory
 *            access attribute, as on coherent CPU-GPU links), every row
 *            buffer and output is page-locked memory mapped into the device's
 *            address space (cudaHostAlloc / cudaHostRegister), and rows are
 *            16-byte aligned: gamma and beta are copied to the workspace and
 *            the kernel reads X, R and writes the outputs in place over the
 *            host link, with 16-byte loads and stores only (no bulk copies),
 *            all on `stream` (kernels and at most two copies: the call can
 *            be captured into a CUDA graph);
 *   pipelined otherwise: rows go through in chunks of about 4 MiB of X,
 *            pipelined over a copy-in stream, `stream` and a copy-out stream
 *            (created once per device on the first call, which should come
 *            before any stream capture), so both copy directions and the
 *            kernels overlap; each copy is one cudaMemcpyAsync.  Pageable
 *            host memory is correct here but slower.
 * y_host and resid_out_host may equal x_host or r_host exactly (in place);
 * any other overlap is ADDLN_ERR_ALIAS.  Results are those of
 * add_layernorm_fwd on the same rows.  Errors as add_layernorm_fwd, plus
 * ADDLN_ERR_WORKSPACE.  Calls on one device are serialised while they queue
 * their work; they are safe from several host threads.
 */
int add_layernorm_fwd_host(const void *x_host, const void *r_host, const float *gamma_host,
                           const float *beta_host, void *y_host, void *resid_out_host,
                           float *mean_host, float *rstd_host, int64_t rows, int64_t H, float eps,
                           int dtype, void *workspace, int64_t workspace_bytes, void *stream);

/* Device workspace bytes add_layernorm_fwd_host needs (0 for rows == 0), or
 * a negative code for an invalid shape or dtype. */
int64_t add_layernorm_fwd_host_workspace_size(int64_t rows, int64_t H, int dtype, int want_resid,
                                              int want_stats);

/* How the last add_layernorm_fwd_host call that queued work (on any thread)
 * moved its data: ADDLN_HOST_MAPPED, ADDLN_HOST_PIPELINED, or 0 before any
 * such call.  A diagnostic for tests and benchmarks. */
#define ADDLN_HOST_PIPELINED 1
#define ADDLN_HOST_MAPPED 2
int add_layernorm_fwd_host_last_mode(void);

/*
 * Unfused baseline, step 1: A = X + R rounded to dtype, elementwise over n
 * contiguous elements ("算子融合的收益量化" section 1, the separate Residual
 * Add kernel: two reads, one write).  a may equal x or r exactly.
 */
int add_fwd(const void *x, const void *r, void *a, int64_t n, int dtype, void *stream);

/*
 * Unfused baseline, step 2: LayerNorm of the stored A ("算子融合与Kernel合并"
 * 4.2 applied to the [rows, H] tensor a).  Same contract as add_layernorm_fwd
 * without R; mean and rstd may be NULL.  y may equal a exactly.
 */
int layernorm_fwd(const void *a, const float *gamma, const float *beta, void *y, float *mean,
                  float *rstd, int64_t rows, int64_t H, float eps, int dtype, void *stream);

/*
 * Fused row softmax ("算子融合与Kernel合并" 4.3, fused_softmax: a max reduce,
 * an exp-sum reduce and a divide, here with one read of the row from memory
 * and one write):
 *     Y_ij = exp(X_ij - max_j X_ij) / sum_k exp(X_ik - max_j X_ij)
 *   x  [rows, H] input in dtype (required)
 *   y  [rows, H] output in dtype (required); may be x exactly (in place)
 * Arithmetic in fp32 with the hardware base-2 exponential (exp(d) as
 * 2^(d log2 e), results below 2^-126 flushed to zero; CUDA's __expf on rows
 * that are not 16-byte aligned): relative error below 1e-5 wherever the
 * result exceeds 1e-30; Y rounded to nearest even.  Same conventions and
 * error codes as add_layernorm_fwd.
 */
int softmax_fwd(const void *x, void *y, int64_t rows, int64_t H, int dtype, void *stream);

/*
 * Fused bias + GELU + residual (the BiasAdd -> GELU -> Residual chain of the
 * diagram in "算子融合的收益量化", three kernels fused into one):
 *     Y_ij = GELU(X_ij + bias_j) + R_ij,  GELU(v) = v/2 * (1 + erf(v / sqrt 2))
 *   x, r  [rows, H] inputs in dtype (required)
 *   bias  [H] fp32 (required)
 *   y     [rows, H] output in dtype; may be x or r exactly (in place)
 * fp32 arithmetic; erf by Abramowitz and Stegun's formula 7.1.26 (absolute
 * error below 1.5e-7); Y rounded to nearest even.  One read of X and R, one
 * write of Y.  Same conventions and error codes as the calls above.
 */
int bias_gelu_residual_fwd(const void *x, const void *r, const float *bias, void *y,
                           int64_t rows, int64_t H, int dtype, void *stream);

/* Unfused chain, step 1 (the diagram's BiasAdd kernel): T = X + bias per
 * column, [rows, H] in dtype; t may be x exactly. */
int bias_add_fwd(const void *x, const float *bias, void *t, int64_t rows, int64_t H, int dtype,
                 void *stream);

/* Unfused chain, step 2 (the diagram's GELU kernel): U = GELU(T) over n
 * contiguous elements; u may be t exactly.  Step 3 (Residual) is add_fwd. */
int gelu_fwd(const void *t, void *u, int64_t n, int dtype, void *stream);

/*
 * Backward of add_layernorm_fwd.  The pages give no backward (fusion of
 * automatic differentiation is only named as a direction in "CUDA算子融合优化"
 * section 5); this is the textbook derivative of the definition above.  Per row
 * i, with xhat = (A - mean) * rstd and g = dY * gamma:
 *     dA = rstd * (g - (1/H) sum_j g - xhat * (1/H) sum_j g xhat) + dA_in
 *     dX = dR = dA                              (written once, to dx)
 * and over all rows dgamma = sum_i dY xhat, dbeta = sum_i dY.
 *   dy         [rows, H] upstream gradient in dtype (required)
 *   a          [rows, H] the stored sum A (resid_out of the forward), dtype
 *   mean, rstd [rows] fp32, as saved by the forward
 *   gamma      [H] fp32
 *   dres       [rows, H] gradient reaching A from elsewhere (A is also the
 *              residual stream), or NULL
 *   dx         [rows, H] output in dtype; may be dy, a or dres exactly
 *   dgamma, dbeta [H] fp32 outputs, both or neither (NULL: not computed)
 *   workspace  device scratch of at least add_layernorm_bwd_workspace_size()
 *              bytes, 16-byte aligned, owned by the caller; needed only with
 *              dgamma / dbeta.  Holds per-CTA column partials, summed in a
 *              fixed order, so the results are bitwise reproducible from
 *              call to call for a shape on one GPU model (the number of
 *              partials follows the SM count and occupancy, so another
 *              model may round the sums differently).  Its
 *              contents need no initialisation; calls that may overlap on
 *              the GPU must not share a workspace.
 * rows == 0 zero-fills dgamma and dbeta.  fp32 arithmetic; dx rounded to
 * nearest even.  Returns ADDLN_OK, or a negative code (ADDLN_ERR_WORKSPACE
 * for a missing, short or misaligned workspace).
 */
int add_layernorm_bwd(const void *dy, const void *a, const float *mean, const float *rstd,
                      const float *gamma, const void *dres, void *dx, float *dgamma, float *dbeta,
                      int64_t rows, int64_t H, int dtype, void *workspace, int64_t workspace_bytes,
                      void *stream);

/* Bytes of workspace add_layernorm_bwd needs for rows x H in dtype on the
 * current device (0 when rows == 0): the larger of what 16-byte-aligned and
 * unaligned rows need, counting only the kinds of rows the library can run
 * at this H.  A negative code on error. */
int64_t add_layernorm_bwd_workspace_size(int64_t rows, int64_t H, int dtype);

/* Size of the built-in scratch buffer add_layernorm_bwd_noalloc uses. */
#define ADDLN_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * add_layernorm_bwd without a caller-provided workspace, for callers that
 * cannot allocate device memory: e.g. a plugin that a framework or inference
 * engine gives only tensor pointers (the host owns all device memory and
 * offers no allocator), or a latency-critical loop where cudaMalloc/cudaFree
 * are ruled out because they can block and synchronise.  The source pages
 * have no counterpart: this is a deployment convenience, not part of the
 * method.
 *
 * Same arguments, results and error codes as add_layernorm_bwd, minus the
 * workspace.  The column partials go to a device buffer of
 * ADDLN_NOALLOC_SCRATCH_BYTES (32 MiB) compiled into the library, which every
 * GPU that loads the library keeps until the process exits.  No device memory
 * is allocated by the call.  The first call on each device that computes
 * dgamma / dbeta looks up the buffer's device address (cudaGetSymbolAddress)
 * with that device current, and caches it for the device's current context
 * (after cudaDeviceReset the new context's address is looked up again); make
 * that first call before any stream capture.  Argument errors are reported
 * with the same codes, checked in the same order, as add_layernorm_bwd.  A
 * shape whose workspace would exceed the buffer
 * (add_layernorm_bwd_workspace_size() > ADDLN_NOALLOC_SCRATCH_BYTES) is
 * rejected with ADDLN_ERR_WORKSPACE before any launch.  All calls on a
 * device share the buffer, which keeps the last call's contents (nothing in
 * it needs to start at zero): calls that may overlap on the GPU, from other
 * streams or host threads, race on it and must be serialised by the
 * caller.
 */
int add_layernorm_bwd_noalloc(const void *dy, const void *a, const float *mean,
                              const float *rstd, const float *gamma, const void *dres, void *dx,
                              float *dgamma, float *dbeta, int64_t rows, int64_t H, int dtype,
                              void *stream);

/* Static text for a return code (never NULL). */
const char *addln_strerror(int code);

/* Largest H accepted for dtype (32768 for 16-bit types, 16384 for fp32), or
 * ADDLN_ERR_DTYPE. */
int64_t addln_max_hidden(int dtype);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * words, which a kernel (add-LayerNorm, softmax or backward) sets when a bounded wait
 * on its own TMA copy runs out.
 * Returns ADDLN_OK, ADDLN_ERR_DEVICE_TIMEOUT, or ADDLN_ERR_CUDA if the
 * synchronisation or the read failed.  Rows of a kernel that timed out are
 * left unwritten.  In the bounds-checked build (see addln_bounds_checked) it
 * also reads and clears the words in which kernels record the first global
 * access they skipped for falling outside its buffer, and returns
 * ADDLN_ERR_BOUNDS if any did (details: addln_bounds_violation).
 */
int addln_get_device_error(void *stream);

/*
 * 1 if this library was built with ADDLN_CHECK_BOUNDS defined, else 0.  In
 * that build every global load, store, bulk copy and L2 prefetch of every
 * kernel is first tested against the extent of the buffer it addresses
 * (from the call's rows, H, dtype and grid); an access that would leave its
 * buffer is skipped, not made, so the context stays usable, and is reported
 * by addln_get_device_error.  A debugging build: slower, and its outputs are
 * not valid once a violation was reported.  The normal build compiles every
 * test away.  No counterpart on the source pages.
 */
int addln_bounds_checked(void);

/*
 * Checked build: the word of the last violation addln_get_device_error
 * reported (bit 63 set; bits 48..62 the number of the access site in the
 * kernel sources; bits 0..47 the byte offset that was out of range), or 0.
 */
uint64_t addln_bounds_violation(void);

/*
 * Test and benchmark only.  Forces the kernel path of add_layernorm_fwd,
 * layernorm_fwd and softmax_fwd (ADDLN_PATH_*; softmax has no CTA_VEC path);
 * ADDLN_PATH_AUTO restores the dispatcher.  A
 * forced path that cannot run a call's arguments makes that call return
 * ADDLN_ERR_UNSUPPORTED.  Returns the previous setting, or ADDLN_ERR_SHAPE
 * for an unknown path.
 */
int addln_set_force_path(int path);

/*
 * Test only.  Sets the bound, in nanoseconds, of the waits on in-flight TMA
 * copies (default 1e9).  0 makes every such wait give up at once, which
 * exercises the timeout path without any hang: the kernel records
 * ADDLN_ERR_DEVICE_TIMEOUT, waits (again bounded, 1 s) for its copies to
 * land, and returns.  Returns the previous value.
 */
uint64_t addln_set_wait_limit_ns(uint64_t ns);

/*
 * Test and benchmark only.  Sets the grid of the persistent CTA-per-row
 * kernels to min(ctas, rows) CTAs, which may be more than one wave
 * (0 = one wave of resident CTAs, the default).  Returns the previous value.
 */
int64_t addln_set_grid_cap(int64_t ctas);

/*
 * Test and benchmark only.  Programmatic dependent launch (default 1 = on):
 * every kernel is launched with programmatic stream serialisation, lets the
 * next kernel in the stream begin launching once all its CTAs run, and waits
 * for the previous kernel's completion before its first global memory
 * access, so stream order and data dependences are kept.  0 launches plainly.
 * Returns the previous setting.
 */
int addln_set_pdl(int on);

/*
 * Test and benchmark only.  Shape of the TMA CTA-per-row kernel: `threads`
 * per CTA (128, 256 or 512; 16-bit rows of at most 4096 elements; 0 =
 * chosen from H) and `stages` rows staged per CTA (1..4; 0 = chosen from the
 * registers and shared memory the kernel takes).  A shape that cannot run a call makes it return
 * ADDLN_ERR_UNSUPPORTED.  Returns the previous thread setting, or
 * ADDLN_ERR_SHAPE for a value out of range.
 */
int addln_set_cta_shape(int threads, int stages);

/*
 * Test and benchmark only.  Rows each warp takes on the warp-per-row vector
 * path of add_layernorm_fwd / layernorm_fwd (rows of up to 1024 elements):
 * 0 (default) = two for rows of 3 or 4 16-byte vectors a lane when the call
 * has at least 16 rows per SM, else one; 1 or 2 forces it (rows of other
 * lengths always take one).  Returns the previous setting, or
 * ADDLN_ERR_SHAPE for another value.
 */
int addln_set_warp_rows(int rows);

/* Name of the kernel path the last add_layernorm_fwd / layernorm_fwd call on
 * this host thread launched (static text; "none" before the first launch). */
const char *addln_last_path(void);

/* Text of the CUDA runtime error behind the last ADDLN_ERR_LAUNCH returned on
 * this host thread (static text; "none" if there was none). */
const char *addln_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ADDLN_H */
