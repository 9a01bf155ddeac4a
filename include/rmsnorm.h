/*
 * rmsnorm.h -- C ABI of the GB300 (sm_103a) row-wise RMSNorm library.
 *
 * Operation ("Pre-built kernel library guide" (FlyDSL), section 1.2 RMSNorm):
 * for every row i of an M x N row-major matrix,
 *     rstd_i = 1 / sqrt(mean_j(x_ij^2) + eps)
 *     y_ij   = x_ij * rstd_i * gamma_j
 * with fp32 accumulation and one final round-to-nearest-even to the output
 * dtype.  The same section names the optional per-row rstd output read by the
 * backward (eps folded into it) and fp32 weights with 16-bit activations.
 *
 * Conventions shared by every entry point:
 *  - Pointers are DEVICE pointers owned by the caller.  The library never
 *    allocates, frees or synchronises; work is enqueued on `stream` (0 = the
 *    legacy default stream) of the current device.  The compute calls may
 *    therefore be captured into a CUDA graph (stream capture) once a call of
 *    the same shape has run outside capture on that device (the first call
 *    sets kernel attributes); rmsnorm_check_device synchronises and may not.
 *  - Layout: contiguous row-major, row stride N elements.
 *  - Dtypes: output dtype = x_dtype; rstd and dgamma are always fp32.
 *    Supported (x_dtype, w_dtype) pairs: (F32, F32), (BF16, BF16), (BF16, F32).
 *  - Alignment: each pointer must be aligned to its element size; 16-byte
 *    alignment of the rows is NOT required.  RMSNorm rows that do not start
 *    on 16 bytes, or inputs (x, dy) whose start differs modulo 16 from the
 *    outputs', take vectorised kernels with scalar row ends (slower than
 *    aligned rows); outputs that disagree with each other modulo 16 (y and
 *    the fused add's residual, dx and dres) take a scalar path.
 *  - Sizes: M == 0 returns RMSNORM_OK without launching; M < 0, N < 1,
 *    N > 2^30, or eps < 0 / NaN return RMSNORM_ERR_INVALID_ARG.
 *  - Aliasing: only fused-add's `residual` is in-out.  Any other overlap of
 *    an output with another operand returns RMSNORM_ERR_INVALID_ARG.
 *  - Errors: a status is returned, no exception crosses the ABI, the device
 *    never traps.  Argument errors launch nothing.  RMSNORM_ERR_CUDA means a
 *    CUDA call failed (the sticky error of `cudaGetLastError` is consumed).
 *  - Non-finite inputs propagate (a zero row with eps = 0 gives NaN).
 */
#ifndef RMSNORM_GB300_H
#define RMSNORM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same declaration as the CUDA runtime's, so either header may come first. */
typedef struct CUstream_st* cudaStream_t;

typedef enum rmsnorm_dtype {
  RMSNORM_F32 = 0,  /* IEEE binary32 */
  RMSNORM_BF16 = 1  /* bfloat16 (upper half of binary32) */
} rmsnorm_dtype_t;

typedef enum rmsnorm_status {
  RMSNORM_OK = 0,
  RMSNORM_ERR_INVALID_ARG = 1,       /* bad size, NULL pointer, overlap, eps */
  RMSNORM_ERR_UNSUPPORTED_DTYPE = 2, /* (x_dtype, w_dtype) pair not supported */
  RMSNORM_ERR_MISALIGNED = 3,        /* pointer not aligned to its element size */
  RMSNORM_ERR_WORKSPACE = 4,         /* backward workspace NULL or too small */
  RMSNORM_ERR_CUDA = 5,              /* a CUDA runtime call failed */
  RMSNORM_ERR_TIMEOUT = 6            /* rmsnorm_check_device: a bounded wait gave up */
} rmsnorm_status_t;

/*
 * Forward.  x: M x N (x_dtype), gamma: N (w_dtype), y: M x N (x_dtype).
 * rstd: M fp32, or NULL to skip it.  Reads x and gamma once, writes y (and
 * rstd).
 */
rmsnorm_status_t rmsnorm_fwd(const void* x, const void* gamma, void* y, float* rstd,
                             int64_t M, int64_t N, float eps, rmsnorm_dtype_t x_dtype,
                             rmsnorm_dtype_t w_dtype, cudaStream_t stream);

/*
 * Fused residual add + forward (the fused-add variant listed in "TIRx
 * kernels", Kernels list, flashinfer.norm ports).  Per element
 *     h_ij = round_xdtype(residual_ij + x_ij)      written over residual
 *     y_ij = RMSNorm(h)_ij * gamma_j               (of the stored, rounded h)
 * x: M x N (read only); residual: M x N, in: r, out: h; gamma: N; y: M x N;
 * rstd: M fp32 of h, or NULL.
 */
rmsnorm_status_t rmsnorm_fused_add_fwd(const void* x, void* residual, const void* gamma,
                                       void* y, float* rstd, int64_t M, int64_t N, float eps,
                                       rmsnorm_dtype_t x_dtype, rmsnorm_dtype_t w_dtype,
                                       cudaStream_t stream);

/*
 * Forward over strided rows: the per-head q/k RMSNorm ("TIRx kernels", Kernels
 * list, flashinfer.norm: qk_rmsnorm).  Row (t, h) of a [T, H, D] view starts
 * at element t * x_stride_token + h * x_stride_head of x (its D elements
 * contiguous) and is written at t * y_stride_token + h * y_stride_head of y;
 * every row is normalised over D with the same gamma (D values).  Strides are
 * in elements and non-negative; the rows of one view must not overlap
 * (x_stride_head >= D when H > 1, x_stride_token >= (H-1) * x_stride_head + D
 * when T > 1).  This covers q or k as a slice of a fused QKV projection output
 * (x_stride_token = row width of that output, x_stride_head = D).  y may be x
 * with the same strides (in place); otherwise the two views must not overlap.
 * rstd: T * H fp32 (row t * H + h), or NULL.  Rows whose starts and strides
 * are 16-byte aligned take the vectorised path; any other layout is handled
 * by a scalar path.
 */
rmsnorm_status_t rmsnorm_fwd_strided(const void* x, int64_t x_stride_token,
                                     int64_t x_stride_head, const void* gamma, void* y,
                                     int64_t y_stride_token, int64_t y_stride_head, float* rstd,
                                     int64_t T, int64_t H, int64_t D, float eps,
                                     rmsnorm_dtype_t x_dtype, rmsnorm_dtype_t w_dtype,
                                     cudaStream_t stream);

/*
 * LayerNorm forward ("Pre-built kernel library guide", section 1.1):
 *     y_ij = (x_ij - mean_i) * rstd_i * gamma_j + beta_j,
 *     mean_i = (1/N) sum_j x_ij,   rstd_i = 1 / sqrt((1/N) sum_j (x_ij - mean_i)^2 + eps)
 * (two passes: the mean, then the population variance about it).  x: M x N
 * (x_dtype); gamma, beta: N (w_dtype; beta NULL for no shift); y: M x N
 * (x_dtype); mean, rstd: M fp32 each, or NULL to skip.  Buffers must not
 * overlap.  Rows that are 16-byte aligned take the vectorised kernels; any
 * other layout a scalar one.
 */
rmsnorm_status_t layernorm_fwd(const void* x, const void* gamma, const void* beta, void* y,
                               float* mean, float* rstd, int64_t M, int64_t N, float eps,
                               rmsnorm_dtype_t x_dtype, rmsnorm_dtype_t w_dtype,
                               cudaStream_t stream);

/* Bytes of device workspace layernorm_bwd needs for these sizes on `device`
 * (-1: the current device), written to *bytes: the fp32 partial rows of the
 * two weight gradients. */
rmsnorm_status_t layernorm_bwd_workspace_size(int64_t M, int64_t N, rmsnorm_dtype_t x_dtype,
                                              rmsnorm_dtype_t w_dtype, int device,
                                              size_t* bytes);

/*
 * LayerNorm backward.  The pages give no formula; differentiating the forward
 * with xhat = (x - mean) rstd and g = dy * gamma:
 *     dx_ij     = rstd_i (g_ij - (1/N) sum_k g_ik - xhat_ij (1/N) sum_k g_ik xhat_ik)
 *     dgamma_j  = sum_i dy_ij xhat_ij,    dbeta_j = sum_i dy_ij
 * dy, x: M x N (x_dtype); mean, rstd: the forward's saved statistics (M fp32
 * each), or both NULL to recompute them from x and eps (eps is used only
 * then); gamma: N (w_dtype); dx: M x N (x_dtype); dgamma, dbeta: N fp32 each,
 * either may be NULL to skip it.  The weight gradients are deterministic:
 * per-CTA partial rows in `workspace` (at least layernorm_bwd_workspace_size
 * bytes, 16-byte aligned; unused when both are NULL), then a fixed-order sum.
 */
rmsnorm_status_t layernorm_bwd(const void* dy, const void* x, const float* mean,
                               const float* rstd, const void* gamma, void* dx, float* dgamma,
                               float* dbeta, void* workspace, size_t workspace_bytes, int64_t M,
                               int64_t N, float eps, rmsnorm_dtype_t x_dtype,
                               rmsnorm_dtype_t w_dtype, cudaStream_t stream);

/*
 * Forward with FP8 output and one scale per row (token): the quantised-output
 * norms named in "TIRx kernels", Kernels list (flashinfer.norm: rmsnorm_quant,
 * fused_add_rmsnorm_quant).  The pages give the names only; this is the plain
 * reading.  With y the forward's output (of x, or, when residual is not
 * NULL, of h = residual + x rounded to x_dtype and written over residual as
 * in rmsnorm_fused_add_fwd):
 *     scale_i = max_j |y_ij| / 448            fp32, the dequantisation scale
 *     q_ij    = e4m3(y_ij / scale_i)          so y_ij ~ e4m3_value(q_ij) * scale_i
 * e4m3: OCP FP8 E4M3 (no infinities, largest finite 448), round to nearest
 * even, saturating.  A row whose x * gamma (h * gamma) is all zero gets
 * scale 0 and codes 0 for any eps.  x: M x N (x_dtype); residual: M x N or
 * NULL; gamma: N (w_dtype); q: M x N bytes; scale: M fp32; rstd: M fp32 or
 * NULL.  Buffers must not overlap.  Rows that are 16-byte aligned with q
 * 8-byte aligned take the vectorised kernels; any other layout a scalar one.
 */
rmsnorm_status_t rmsnorm_fwd_fp8(const void* x, void* residual, const void* gamma, void* q,
                                 float* scale, float* rstd, int64_t M, int64_t N, float eps,
                                 rmsnorm_dtype_t x_dtype, rmsnorm_dtype_t w_dtype,
                                 cudaStream_t stream);

/*
 * Forward with NVFP4 output: the FP4 norms named in "TIRx kernels", Kernels
 * list (flashinfer.norm: rmsnorm_fp4quant, add_rmsnorm_fp4quant; the format
 * of flashinfer.quantization: nvfp4_quantize).  Plain reading of the names:
 * N must be a multiple of 16; each row splits into blocks of 16 consecutive
 * elements; global_scale (gs) is the caller's per-tensor scale, finite and
 * > 0.  With y as in rmsnorm_fwd_fp8, for block b:
 *     S_b = e4m3(gs * max_b |y| / 6)          stored in block_scale
 *     q_j = e2m1(y_j * gs / S_b)              (0 when S_b = 0)
 * so y_j ~ e2m1_value(q_j) * S_b / gs.  e2m1: FP4 E2M1 (0, 0.5, 1, 1.5, 2,
 * 3, 4, 6), round to nearest even, saturating.  q: M x N/2 bytes, two codes
 * per byte, element 2k in the low nibble; block_scale: M x N/16 E4M3 bytes,
 * row-major (the plain layout, not a tensor-core swizzle).  Other arguments
 * and the fused residual add as in rmsnorm_fwd_fp8.
 */
rmsnorm_status_t rmsnorm_fwd_nvfp4(const void* x, void* residual, const void* gamma,
                                   float global_scale, void* q, void* block_scale, float* rstd,
                                   int64_t M, int64_t N, float eps, rmsnorm_dtype_t x_dtype,
                                   rmsnorm_dtype_t w_dtype, cudaStream_t stream);

/*
 * Workspace of rmsnorm_bwd, in bytes, for these sizes on `device` (-1: the
 * current device).  It depends on the device's SM count, and covers every
 * alignment of the operands (those off 16 bytes may take a kernel with more
 * CTAs, hence more partial rows, than aligned ones).  Writes *bytes (0 when
 * M == 0 or no dgamma is wanted is still a valid answer to pass).
 */
rmsnorm_status_t rmsnorm_bwd_workspace_size(int64_t M, int64_t N, rmsnorm_dtype_t x_dtype,
                                            rmsnorm_dtype_t w_dtype, int device,
                                            size_t* bytes);

/*
 * Backward ("Pre-built kernel library guide", section 1.2: reads the forward's
 * input, gamma, dy and rstd; writes dx and the weight gradient).  With
 *     c_i = rstd_i^2 / N * sum_k gamma_k dy_ik x_ik
 *     dx_ij     = rstd_i * (gamma_j dy_ij - x_ij c_i)         (x_dtype)
 *     dgamma_j  = sum_i dy_ij x_ij rstd_i                      (fp32)
 * dy, x, dx: M x N; gamma: N; rstd: M fp32 from the forward (eps is then
 * ignored), or NULL to recompute it from x and eps.  dgamma: N fp32, or NULL
 * to skip the weight gradient.  dgamma is reduced over the rows in a fixed
 * order through `workspace` (device memory of at least
 * rmsnorm_bwd_workspace_size bytes, 16-byte aligned, contents ignored), so it
 * is bit-for-bit reproducible run to run on the same device.  Two launches on
 * `stream`.
 */
rmsnorm_status_t rmsnorm_bwd(const void* dy, const void* x, const float* rstd,
                             const void* gamma, void* dx, float* dgamma, void* workspace,
                             size_t workspace_bytes, int64_t M, int64_t N, float eps,
                             rmsnorm_dtype_t x_dtype, rmsnorm_dtype_t w_dtype,
                             cudaStream_t stream);

/*
 * Backward of the fused residual add (the fused-add training wrapper of "Pre-
 * built kernel library guide", section 1.2): for h = residual + x and
 * y = RMSNorm(h) * gamma, both the residual and x receive
 *     dh_ij = rstd_i * (gamma_j dy_ij - h_ij c_i) + dres_ij
 * where dres is the gradient that reaches h along the residual path and c_i
 * is as in rmsnorm_bwd (with h in place of x).  h: M x N, the stored sum the
 * forward normalised; rstd: M fp32 from the forward, or NULL to recompute from
 * h and eps; dres: M x N, in: the residual-path gradient, out: dh (x_dtype,
 * rounded once).  dgamma: N values in dgamma_dtype (RMSNORM_F32, or
 * RMSNORM_BF16 rounded once from the fp32 sum -- the weight dtype of a bf16
 * model), or NULL; reduced in a fixed order through `workspace` like
 * rmsnorm_bwd, whose workspace query (rmsnorm_bwd_workspace_size) serves this
 * call too.  Two launches on `stream`.
 */
rmsnorm_status_t rmsnorm_fused_add_bwd(const void* dy, const void* h, const float* rstd,
                                       const void* gamma, void* dres, void* dgamma,
                                       rmsnorm_dtype_t dgamma_dtype, void* workspace,
                                       size_t workspace_bytes, int64_t M, int64_t N, float eps,
                                       rmsnorm_dtype_t x_dtype, rmsnorm_dtype_t w_dtype,
                                       cudaStream_t stream);

/*
 * Backward for callers that cannot allocate device memory.  No counterpart in
 * the source pages: this entry point exists for integration only.
 *
 * Some callers have no way to provide the workspace rmsnorm_bwd needs: a
 * serving runtime that has handed all device memory to its own pool and
 * forbids other allocations, a plugin interface that gives an operator its
 * inputs and outputs but no allocator, or a latency-critical path where a
 * cudaMalloc / cudaFree (which can synchronise the device) is not acceptable.
 * This call computes exactly what rmsnorm_bwd computes, with the same
 * arguments minus the workspace; the dgamma partial rows go to a scratch
 * array of RMSNORM_BWD_NOALLOC_SCRATCH_BYTES that is part of the library's
 * device image.  Neither the library nor the caller allocates anything.
 *
 *  - Limit: a shape whose size from rmsnorm_bwd_workspace_size fits in
 *    RMSNORM_BWD_NOALLOC_SCRATCH_BYTES always runs.  Where it does not, the
 *    call runs when the partial rows of 16-byte aligned operands fit (it
 *    then gives operands at other offsets fewer CTAs than rmsnorm_bwd
 *    would) and is otherwise rejected with RMSNORM_ERR_WORKSPACE before any
 *    launch.
 *  - Memory: every GPU that loads the library keeps the scratch until the
 *    process exits.
 *  - Set-up: the first call on each device looks up the scratch's device
 *    address (cudaGetSymbolAddress, with that device current); make that
 *    first call before any stream capture.
 *  - Sharing: all calls on a device share the one scratch, which keeps the
 *    last call's contents (each call rewrites every part it reads, so nothing
 *    needs clearing).  Calls that overlap on the GPU -- for example on two
 *    streams without ordering between them -- race on it and may return a
 *    wrong dgamma; order them on one stream or with events.
 *  - Lifetime: the looked-up address is kept for the life of the process.
 *    After cudaDeviceReset (or anything else that destroys the device's
 *    primary context) the library's device image -- and so the scratch --
 *    is loaded again at another address; do not call this function on that
 *    device again in the same process.
 */
#define RMSNORM_BWD_NOALLOC_SCRATCH_BYTES (16u << 20)

rmsnorm_status_t rmsnorm_bwd_noalloc(const void* dy, const void* x, const float* rstd,
                                     const void* gamma, void* dx, float* dgamma, int64_t M,
                                     int64_t N, float eps, rmsnorm_dtype_t x_dtype,
                                     rmsnorm_dtype_t w_dtype, cudaStream_t stream);

/*
 * Device-side status of the current device, for the kernels that stream rows
 * through bulk copies (cp.async.bulk) and wait for them on mbarriers.  Every
 * such wait is bounded (about 2 s of SM clock); a kernel whose wait runs out
 * writes nothing more for that row, waits (bounded) for the copies it still
 * has in flight, sets a flag in a device status word and returns, so the
 * context stays usable.  This call waits for `stream` to finish, reads and
 * clears that flag, and returns RMSNORM_ERR_TIMEOUT if it was set, else
 * RMSNORM_OK.  Unlike the other entry points it synchronises (the stream).
 * No page this library follows has this call; it is the error channel of
 * the bounded waits.
 */
rmsnorm_status_t rmsnorm_check_device(cudaStream_t stream);

/*
 * Text naming the CUDA call that failed and its error, for the last
 * RMSNORM_ERR_CUDA returned to the calling thread ("" if none).  The string
 * belongs to the library and stays valid until that thread's next call.
 */
const char* rmsnorm_last_error(void);

/*
 * Re-read the debug and measurement knobs from the environment.  The library
 * reads them once when it is loaded, never while launching:
 *   RMSNORM_FORCE_VARIANT      force a kernel variant (A/B runs, tests); a
 *                              variant that cannot serve a call makes that
 *                              call return RMSNORM_ERR_INVALID_ARG
 *   RMSNORM_WAIT_LIMIT_CYCLES  clock cycles a bulk-copy wait lasts before it
 *                              gives up (negative: give up at once)
 *   RMSNORM_NO_PDL=1           launch without programmatic dependent launch
 * Call it only while no other thread is inside the library.  No page this
 * library follows has this call; it exists for tests and measurements.
 */
void rmsnorm_reload_debug_env(void);

/* Static text of a status code ("unknown status" for other values). */
const char* rmsnorm_status_string(rmsnorm_status_t status);

/*
 * The kernel variant the library would launch for this call shape, as text
 * (for example "fwd/cta/vpt4/t256"), into buf (NUL-terminated, truncated to
 * len).  op: 0 forward, 1 fused add, 2 backward, 3 fused-add backward,
 * 4 strided forward (M = tokens x heads rows of N = D elements), 5 FP8
 * forward, 6 fused-add FP8 forward, 7 NVFP4 forward, 8 fused-add NVFP4,
 * 9 LayerNorm forward, 10 LayerNorm backward (with the forward's mean and
 * rstd given).  aligned16:
 * nonzero when all operand base pointers (and, for op 4, all strides) are
 * 16-byte aligned; for ops 0-3, 2 describes outputs on 16 bytes with x (and
 * dy) off them (for example x a view at an odd element offset).  Returns
 * RMSNORM_OK or an argument error; launches nothing.
 */
rmsnorm_status_t rmsnorm_describe_plan(int op, int64_t M, int64_t N, rmsnorm_dtype_t x_dtype,
                                       rmsnorm_dtype_t w_dtype, int aligned16, int device,
                                       char* buf, size_t len);

#ifdef __cplusplus
}
#endif

#endif /* RMSNORM_GB300_H */
