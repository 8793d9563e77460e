/*
 * fp8lin.h - C ABI of the GB300 (sm_103a) FP8 linear-layer library.
 *
 * The library implements the FP8 linear layer of a training step:
 *   quantizers  - fused amax -> fp32 scale -> saturating round-to-nearest-even
 *                 cast, writing the row-major and the transposed FP8 layout in
 *                 one pass ("Native FP8 MLP reconstruction", implementation
 *                 paragraph: current tensorwise amax, E4M3 inputs/weights, E5M2
 *                 incoming gradients, fused cast emitting ordinary and
 *                 transposed layouts);
 *   weight cache - is_first_microbatch semantics ("FP8 weight caching shows no
 *                 speedup ... under Float8BlockScaling", TransformerEngine
 *                 issue #2852, opening post and maintainer reply);
 *   FP8 GEMMs   - fprop, dgrad and wgrad on tcgen05 tensor cores with fp32
 *                 accumulation and BF16 output (use_fast_accum=False in the
 *                 reconstruction's implementation paragraph).
 *
 * Conventions shared by every call
 *   - Tensors are dense and row-major.  X is [N, K] (tokens x in features),
 *     W is [O, K] (out x in), Y = X W^T is [N, O].  A "colwise" or
 *     "transposed" layout of an [R, C] tensor is the [C, R] array, row-major.
 *   - Every tensor pointer is a DEVICE pointer owned by the caller, 16-byte
 *     aligned, except the host buffers of fp8_linear_step_host.  The library
 *     allocates no device memory; scratch space is the caller's `workspace`
 *     (size from the *_workspace_size queries).
 *   - Every dimension must be a multiple of 16 (TMA row-stride rule).  A
 *     dimension need not be a multiple of 128: the last 128-block of a row,
 *     column or tile is then shorter ("ragged tail") and its amax covers the
 *     elements present.  A zero dimension makes the call a no-op (FP8_OK).
 *   - bf16 tensors are passed as `const void*` (IEEE bfloat16 bit patterns).
 *   - Every call enqueues work on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and returns without synchronising, except
 *     fp8_get_device_status and fp8_host_pipeline_sync (fp8_linear_step_host
 *     enqueues on its pipeline's own streams).  Arguments are validated before anything is
 *     launched: on a non-OK status nothing was enqueued.
 *   - Kernels are launched with programmatic dependent launch: a kernel may
 *     be scheduled while the kernel before it on the same stream drains, and
 *     waits for that kernel's completion before it touches memory, so every
 *     result is that of serial stream order.  FP8LIN_PDL=0 in the
 *     environment (read on the first launch) gives plain launches.
 *   - Calls are not thread-safe with respect to one fp8_weight_cache object.
 *     Other calls may come from several host threads: the per-device launch
 *     settings the library fills in on first use (shared-memory opt-in,
 *     resident CTA counts, SM count) are idempotent, so concurrent first
 *     calls store the same values.  The kernel timing of fp8_profile_begin /
 *     fp8_profile_end and the launch counter are process-wide.
 *
 * Recipes
 *   FP8_RECIPE_TENSORWISE: one current (just-in-time) amax per tensor.
 *   FP8_RECIPE_BLOCK (Float8BlockScaling reading): activations and gradients
 *     use 1x128 blocks along each layout's contiguous dimension, weights use
 *     128x128 tiles.  No amax history in either recipe.
 *   Scale rule (both recipes): scale = fp32(fmax / amax) (IEEE division,
 *   round-to-nearest-even), scale_inv = fp32(1 / scale); fmax = 448 (E4M3) or
 *   57344 (E5M2).  amax == 0 gives scale = scale_inv = 1; a quotient that
 *   overflows gives scale = FLT_MAX.  amax ignores NaN.  The cast is one fp32
 *   multiply x * scale, then saturating round-to-nearest-even to 8 bits;
 *   NaN encodes to 0x7F.
 *
 * Scale array shapes (float32, row-major), for an [R, C] input
 *   tensorwise        : rowwise [1], colwise [1] (same value)
 *   1x128 (act, grad) : rowwise [R, ceil(C/128)], colwise [C, ceil(R/128)]
 *   128x128 (weight)  : rowwise [ceil(R/128), ceil(C/128)], colwise = its transpose
 */
#ifndef FP8LIN_H
#define FP8LIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *fp8_stream_t; /* same type as cudaStream_t */

typedef enum {
  FP8_OK = 0,
  FP8_ERR_INVALID_ARG = 1, /* null pointer where one is required, bad enum, negative size */
  FP8_ERR_SHAPE = 2,       /* a dimension not a multiple of 16, or inconsistent shapes */
  FP8_ERR_ALIGN = 3,       /* a device pointer not 16-byte aligned */
  FP8_ERR_STALE = 4,       /* weight-cache entry not quantized in this cycle, or its version changed */
  FP8_ERR_TIMEOUT = 5,     /* a device-side wait gave up (reported by fp8_get_device_status) */
  FP8_ERR_CUDA = 6,        /* a CUDA runtime call or kernel launch failed */
  FP8_ERR_UNSUPPORTED = 7, /* request this build does not implement */
  FP8_ERR_WORKSPACE = 8    /* workspace smaller than the size query returned */
} fp8_status;

/* FP8_RECIPE_DELAYED: DelayedScaling (TransformerEngine issue #2852, opening
 * post: amax_history state).  Quantization by fp8_quantize_delayed; in a
 * weight cache via fp8_weight_cache_register_delayed; in fp8_linear_fwd/bwd
 * the weight uses its cache entry's history while activations and gradients
 * use current tensorwise scaling.  fp8_quantize itself rejects it. */
typedef enum { FP8_RECIPE_TENSORWISE = 0, FP8_RECIPE_BLOCK = 1, FP8_RECIPE_DELAYED = 2 } fp8_recipe;

/* Operand role: ACT and WEIGHT use E4M3, GRAD uses E5M2 (reconstruction,
 * implementation paragraph).  Under FP8_RECIPE_BLOCK, WEIGHT selects 128x128
 * tiles and ACT/GRAD select 1x128 blocks. */
typedef enum { FP8_ROLE_ACT = 0, FP8_ROLE_WEIGHT = 1, FP8_ROLE_GRAD = 2 } fp8_role;

typedef enum { FP8_FORMAT_E4M3 = 0, FP8_FORMAT_E5M2 = 1 } fp8_format;

/* Scale layouts of the two GEMM operands (see fp8_gemm). */
typedef enum {
  FP8_SCALING_TENSOR = 0,        /* a_scale_inv [1], b_scale_inv [1] */
  FP8_SCALING_1x128_128x128 = 1, /* a [M, ceil(K/128)], b [ceil(N/128), ceil(K/128)] (fprop, dgrad) */
  FP8_SCALING_1x128_1x128 = 2    /* a [M, ceil(K/128)], b [N, ceil(K/128)]          (wgrad)        */
} fp8_scaling;

/* Human-readable name of a status code (static string). */
const char *fp8_status_string(fp8_status s);

/* Number of kernels this library has launched since it was loaded (all
 * devices, all streams).  Host-side counter, incremented once per launch. */
uint64_t fp8_launch_count(void);

/* ------------------------------------------------------------------ quantize
 * fp8_quantize: fused amax -> scale -> cast of a bf16 [rows, cols] tensor,
 * writing the row-major bytes `rowwise_out` [rows, cols] and/or the
 * transposed bytes `colwise_out` [cols, rows] in one pass over the input
 * (tensorwise: one extra read of the input for the global amax).
 *   x              device bf16 [rows, cols]
 *   recipe, role   select format and block shape (see above)
 *   rowwise_out    device u8 [rows, cols] or NULL
 *   colwise_out    device u8 [cols, rows] or NULL (not both NULL)
 *   row_scale, row_scale_inv  device f32, rowwise scale shape; required
 *                  when rowwise_out != NULL, and always for tensorwise
 *   col_scale, col_scale_inv  device f32, colwise scale shape; required when
 *                  colwise_out != NULL under 1x128 and 128x128; ignored
 *                  (may be NULL) under tensorwise
 *   workspace      device scratch of fp8_quantize_workspace_size bytes
 *                  (NULL allowed when that size is 0)
 * Errors: INVALID_ARG, SHAPE, ALIGN, WORKSPACE, CUDA.
 */
fp8_status fp8_quantize(const void *x, int64_t rows, int64_t cols, fp8_recipe recipe, fp8_role role,
                        uint8_t *rowwise_out, uint8_t *colwise_out, float *row_scale,
                        float *row_scale_inv, float *col_scale, float *col_scale_inv,
                        void *workspace, size_t workspace_bytes, fp8_stream_t stream);

fp8_status fp8_quantize_workspace_size(fp8_recipe recipe, int64_t rows, int64_t cols,
                                       size_t *bytes);

/* fp8_quantize_delayed: DelayedScaling, margin 0 (one pass over x).
 *   scale = fp32(fmax / max(amax_history[0 .. history_len-1])) with the scale
 *   rule's special cases (an all-zero history gives scale 1); x is cast with
 *   it into rowwise_out [rows, cols] and/or colwise_out [cols, rows]; then
 *   amax(x) is written to amax_history[step % history_len].  scale and
 *   scale_inv receive one float each.  amax_history is caller-owned device
 *   memory (zeros before the first call); workspace as for tensorwise
 *   fp8_quantize_workspace_size.  Errors: INVALID_ARG, SHAPE, ALIGN, WORKSPACE, CUDA. */
fp8_status fp8_quantize_delayed(const void *x, int64_t rows, int64_t cols, fp8_role role,
                                uint8_t *rowwise_out, uint8_t *colwise_out, float *scale,
                                float *scale_inv, float *amax_history, int32_t history_len,
                                int64_t step, void *workspace, size_t workspace_bytes,
                                fp8_stream_t stream);

/* Shape [srows, scols] of the scale array of a layout (colwise = 0 or 1). */
fp8_status fp8_scale_shape(fp8_recipe recipe, fp8_role role, int64_t rows, int64_t cols,
                           int colwise, int64_t *srows, int64_t *scols);

/* ------------------------------------------------------------------ GEMM
 * fp8_gemm: C[M, N] (bf16) = sum_k (A[m, k] * sa) * (B[n, k] * sb), both
 * operands K-major (row-major [M, K] and [N, K] bytes).  sa, sb are the
 * scale_inv values of each element's block under `scaling`.  The tensor
 * cores accumulate in fp32; under the block scalings every 128-deep K block
 * is accumulated separately and added, scaled, into an fp32 accumulator.
 * The result is rounded once to bf16 (round-to-nearest-even).
 *   a_fmt, b_fmt   FP8 format of each operand (E4M3 or E5M2, may differ)
 *   workspace      device scratch, fp8_gemm_workspace_size bytes (split-K
 *                  partial sums; 0 when no split is used)
 * Deterministic: the kernel configuration, split and summation order are a
 * function of (M, N, K, scaling) only.
 * Errors: INVALID_ARG, SHAPE, ALIGN, WORKSPACE, CUDA.
 */
fp8_status fp8_gemm(const uint8_t *A, fp8_format a_fmt, const float *a_scale_inv,
                    const uint8_t *B, fp8_format b_fmt, const float *b_scale_inv, int64_t M,
                    int64_t N, int64_t K, fp8_scaling scaling, void *C, void *workspace,
                    size_t workspace_bytes, fp8_stream_t stream);

fp8_status fp8_gemm_workspace_size(int64_t M, int64_t N, int64_t K, fp8_scaling scaling,
                                   size_t *bytes);

/* ------------------------------------------------------------------ weight cache
 * is_first_microbatch semantics (TransformerEngine issue #2852, opening post;
 * maintainer reply: under non-delayed recipes cached and uncached runs are
 * exactly equal and caching saves the weight re-quantization).
 *   begin_cycle  = start of a gradient-accumulation cycle: every entry becomes
 *                  stale, so the next get() with use_cache re-quantizes
 *                  (is_first_microbatch=True);
 *   get(use_cache=1) on a fresh entry reuses the FP8 copy
 *                  (is_first_microbatch=False);
 *   get(use_cache=0) always re-quantizes (is_first_microbatch=None).
 * The cache is a host object; the FP8 buffers it fills are caller-owned
 * device memory registered once per weight.
 */
typedef struct fp8_weight_cache fp8_weight_cache;
typedef int32_t fp8_weight_handle;

fp8_status fp8_weight_cache_create(fp8_weight_cache **out);
void fp8_weight_cache_destroy(fp8_weight_cache *cache);

/* Register the bf16 weight W [O, K] and the caller-owned buffers that will
 * hold its FP8 copy: w_row [O, K], w_col [K, O] and their scale arrays
 * (weight role shapes under `recipe`).  `workspace` (size from
 * fp8_quantize_workspace_size(recipe, O, K)) must stay valid for every get()
 * of this handle.  Errors: INVALID_ARG, SHAPE, ALIGN, WORKSPACE. */
fp8_status fp8_weight_cache_register(fp8_weight_cache *cache, const void *w, int64_t O,
                                     int64_t K, fp8_recipe recipe, uint8_t *w_row,
                                     uint8_t *w_col, float *row_scale, float *row_scale_inv,
                                     float *col_scale, float *col_scale_inv, void *workspace,
                                     size_t workspace_bytes, fp8_weight_handle *out);

/* Register a weight under DelayedScaling: one tensorwise scale (scale,
 * scale_inv: one float each, shared by both layouts) and a caller-owned
 * amax_history ring of history_len floats (zeros initially).  Every
 * quantization get() performs advances the ring by one position, so
 * re-quantizing inside a cycle (use_cache = 0) is not bitwise neutral. */
fp8_status fp8_weight_cache_register_delayed(fp8_weight_cache *cache, const void *w, int64_t O,
                                             int64_t K, uint8_t *w_row, uint8_t *w_col,
                                             float *scale, float *scale_inv, float *amax_history,
                                             int32_t history_len, void *workspace,
                                             size_t workspace_bytes, fp8_weight_handle *out);

fp8_status fp8_weight_cache_begin_cycle(fp8_weight_cache *cache);

/* Make the FP8 copy of weight `h` current on `stream`.  w_version is a
 * caller-maintained counter of the bf16 weight's contents: get() with
 * use_cache on an entry already quantized in this cycle under another
 * version returns FP8_ERR_STALE (the weight changed mid-cycle).
 * *requantized (optional) is set to 1 when a quantization was enqueued. */
fp8_status fp8_weight_cache_get(fp8_weight_cache *cache, fp8_weight_handle h, uint64_t w_version,
                                int use_cache, fp8_stream_t stream, int *requantized);

/* ------------------------------------------------------------------ linear layer
 * The backward policy follows the implementation paragraph of "Native FP8
 * MLP reconstruction": the forward's rounded FP8 X and W are reused by the
 * backward GEMMs, the incoming gradient is rounded on its own (E5M2), the
 * scales are detached (no gradient flows through them), and every GEMM
 * accumulates in fp32 (use_fast_accum=False) and writes BF16.
 * fp8_linear_fwd: Y[N, O] = X W^T with X quantized (E4M3, both layouts) and
 * the cached FP8 weight; writes Y (bf16) and the context the backward needs
 * (the transposed FP8 X and its scales) into `ctx`.
 * fp8_linear_bwd: dY[N, O] is quantized separately (E5M2, both layouts);
 * dX[N, K] = dY W (dgrad, forward-rounded W reused; dX may be NULL) and
 * dW[O, K] = dY^T X (wgrad, forward-rounded X from ctx reused).  Scales are
 * constants of the backward (detached).
 * The weight handle must have been made current by fp8_weight_cache_get in
 * the current cycle (else FP8_ERR_STALE) and `recipe` must equal its
 * registered recipe (else FP8_ERR_INVALID_ARG).
 *   ctx  device buffer of fp8_linear_ctx_size bytes, written by fwd, read by bwd
 *   ws   device scratch of fp8_linear_workspace_size bytes (shared by fwd and bwd)
 */
fp8_status fp8_linear_ctx_size(fp8_recipe recipe, int64_t N, int64_t K, size_t *bytes);
fp8_status fp8_linear_workspace_size(fp8_recipe recipe, int64_t N, int64_t K, int64_t O,
                                     size_t *bytes);
fp8_status fp8_linear_fwd(const void *X, int64_t N, int64_t K, fp8_weight_cache *cache,
                          fp8_weight_handle h, fp8_recipe recipe, void *Y, void *ctx, void *ws,
                          size_t ws_bytes, fp8_stream_t stream);
fp8_status fp8_linear_bwd(const void *dY, int64_t N, int64_t O, const void *ctx,
                          fp8_weight_cache *cache, fp8_weight_handle h, fp8_recipe recipe,
                          void *dX, void *dW, void *ws, size_t ws_bytes, fp8_stream_t stream);

/* ------------------------------------------------------------------ split tensorwise passes
 * Current tensorwise scaling is two passes over a tensor: per-CTA maxima of
 * |x|, then the cast with scale = fmax / (maximum of those partials).  The
 * first pass reads the whole tensor and nothing else, and its CTAs need almost
 * no shared memory, so it can run on another stream beside a GEMM or a cast
 * on the same GPU.
 *   fp8_amax_partials: the first pass alone over bf16 x [rows, cols], into
 *     `partials` (device, fp8_quantize_workspace_size(TENSORWISE, rows, cols)
 *     bytes, 16-byte aligned; the contents are the library's own format).
 *   fp8_linear_fwd_after_amax / fp8_linear_bwd_after_amax: fp8_linear_fwd /
 *     fp8_linear_bwd whose X (resp. dY) quantization runs only the cast,
 *     reading partials that fp8_amax_partials wrote for that same tensor.
 *     The caller orders the two (e.g. an event between the streams).
 *     Tensorwise and delayed recipes (their activations use current
 *     tensorwise scaling); the block recipe returns FP8_ERR_UNSUPPORTED.
 * Results are bit for bit those of fp8_linear_fwd / fp8_linear_bwd.
 * Errors: as fp8_linear_fwd / bwd and fp8_quantize (WORKSPACE for a short
 * partials buffer). */
fp8_status fp8_amax_partials(const void *x, int64_t rows, int64_t cols, void *partials,
                             size_t partials_bytes, fp8_stream_t stream);
fp8_status fp8_linear_fwd_after_amax(const void *X, const void *x_partials, int64_t N, int64_t K,
                                     fp8_weight_cache *cache, fp8_weight_handle h,
                                     fp8_recipe recipe, void *Y, void *ctx, void *ws,
                                     size_t ws_bytes, fp8_stream_t stream);
fp8_status fp8_linear_bwd_after_amax(const void *dY, const void *dy_partials, int64_t N, int64_t O,
                                     const void *ctx, fp8_weight_cache *cache, fp8_weight_handle h,
                                     fp8_recipe recipe, void *dX, void *dW, void *ws,
                                     size_t ws_bytes, fp8_stream_t stream);

/* ------------------------------------------------------------------ fused producers
 * Quantization fused into the producer of the quantized tensor (block recipe
 * only; other recipes return FP8_ERR_UNSUPPORTED).  The bf16 intermediate is
 * never written: each kernel computes it in fp32, rounds it to bf16 exactly
 * as fp8_gelu_fwd / fp8_gelu_bwd do, and quantizes that value, so the bytes
 * and scales equal those of the unfused sequence bit for bit.
 *   fp8_gelu_quantize:     A = bf16(GELU(H)), 1x128 E4M3 (activation role)
 *   fp8_gelu_bwd_quantize: dH = bf16(dA * GELU'(H)), 1x128 E5M2 (gradient role)
 * Output arguments as in fp8_quantize (both layouts optional, not both NULL).
 * Errors: UNSUPPORTED, INVALID_ARG, SHAPE, ALIGN, CUDA. */
fp8_status fp8_gelu_quantize(const void *H, int64_t rows, int64_t cols, fp8_recipe recipe,
                             uint8_t *rowwise_out, uint8_t *colwise_out, float *row_scale,
                             float *row_scale_inv, float *col_scale, float *col_scale_inv,
                             fp8_stream_t stream);
fp8_status fp8_gelu_bwd_quantize(const void *dA, const void *H, int64_t rows, int64_t cols,
                                 fp8_recipe recipe, uint8_t *rowwise_out, uint8_t *colwise_out,
                                 float *row_scale, float *row_scale_inv, float *col_scale,
                                 float *col_scale_inv, fp8_stream_t stream);

/* Linear layer on operands quantized by the caller (e.g. by a fused producer).
 * fp8_linear_ctx_layout returns where, inside a linear context buffer, the
 * transposed FP8 input and its scale arrays live, so a producer can write the
 * saved operand directly.  fp8_linear_fwd_quantized = the fprop GEMM of
 * fp8_linear_fwd with X given as its rowwise bytes and scale_inv (the caller
 * has already filled the context's transposed part); fp8_linear_bwd_quantized
 * = the dgrad (dX may be NULL) and wgrad GEMMs of fp8_linear_bwd with dY
 * given in both layouts.  Same weight-cache and recipe rules as the bf16 calls. */
fp8_status fp8_linear_ctx_layout(fp8_recipe recipe, int64_t N, int64_t K, void *ctx,
                                 uint8_t **xq_col, float **col_scale, float **col_scale_inv);
fp8_status fp8_linear_fwd_quantized(const uint8_t *xq_row, const float *xq_row_scale_inv,
                                    int64_t N, int64_t K, fp8_weight_cache *cache,
                                    fp8_weight_handle h, fp8_recipe recipe, void *Y, void *ws,
                                    size_t ws_bytes, fp8_stream_t stream);
fp8_status fp8_linear_bwd_quantized(const uint8_t *gq_row, const float *gq_row_scale_inv,
                                    const uint8_t *gq_col, const float *gq_col_scale_inv,
                                    int64_t N, int64_t O, const void *ctx, fp8_weight_cache *cache,
                                    fp8_weight_handle h, fp8_recipe recipe, void *dX, void *dW,
                                    void *ws, size_t ws_bytes, fp8_stream_t stream);

/* ------------------------------------------------------------------ MLP glue
 * GELU in its exact erf form, fp32 arithmetic, bf16 in/out, n elements
 * (n a multiple of 8): A = H * Phi(H); dH = dA * (Phi(H) + H * phi(H)).
 * fp8_grad_accumulate: acc[i] += float(dW[i]) in fp32 (one add per element),
 * for gradient accumulation over microbatches. */
fp8_status fp8_gelu_fwd(const void *H, void *A, int64_t n, fp8_stream_t stream);
fp8_status fp8_gelu_bwd(const void *dA, const void *H, void *dH, int64_t n, fp8_stream_t stream);
fp8_status fp8_grad_accumulate(float *acc, const void *dW, int64_t n, fp8_stream_t stream);

/* ------------------------------------------------------------------ host-buffer steps
 * One forward + backward of an isolated FP8 linear (fp8_linear_fwd then
 * fp8_linear_bwd, same recipe rules) whose inputs and results live in HOST
 * memory: the library copies them to and from the caller's device buffers.
 * Host buffers should be page-locked (cudaHostAlloc / pinned): pageable
 * memory works but then the copies stage through the CUDA driver and block.
 *
 * A pipeline owns three CUDA streams on the device current at creation
 * (copy-in, compute, copy-out) and `slots` sets of events.  Each slot stands
 * for one set of device buffers (one linear).  fp8_linear_step_host(slot):
 *   copy-in:  X, W host -> device (W into the buffer registered for the
 *             weight handle) once this slot's previous forward has read them,
 *             then dY once this slot's previous backward has read it;
 *   compute:  fp8_weight_cache_get(h, w_version, use_cache = 1) and
 *             fp8_linear_fwd once X and W are in and this slot's previous Y
 *             has left the device; fp8_linear_bwd once dY is in and this
 *             slot's previous dX and dW have left the device;
 *   copy-out: Y as soon as the forward has finished, then dX (if both
 *             pointers are set) and dW after the backward.
 * So within one call dY streams in while the forward runs and Y streams out
 * while the backward runs.
 * Calls on different slots overlap: the copies of one linear run while
 * another's kernels execute.  The compute work of all slots is ordered on the
 * one compute stream, so `ctx` and `ws` may be shared by all slots; the
 * weight handle of a slot must not be used by another slot.  The call
 * returns once everything is enqueued; results are on the host after
 * fp8_host_pipeline_sync (or after fp8_host_pipeline_join on a stream that
 * is then synchronised).
 *   fp8_host_pipeline_fork(p, s): the pipeline's streams wait for the work
 *     enqueued on s so far (an event recorded on s before marks a start).
 *   fp8_host_pipeline_join(p, s): s waits for all work enqueued on the
 *     pipeline so far (an event recorded on s afterwards marks the end).
 * Errors: INVALID_ARG (null pipeline, slot out of range, null buffer, handle
 * or recipe mismatch), SHAPE, ALIGN (device buffers), STALE, WORKSPACE, CUDA.
 * Nothing is enqueued when a check fails. */
typedef struct fp8_host_pipeline fp8_host_pipeline;
typedef struct {
  const void *X;  /* [N, K] bf16 */
  const void *W;  /* [O, K] bf16 */
  const void *dY; /* [N, O] bf16 */
  void *Y;        /* [N, O] bf16 */
  void *dX;       /* [N, K] bf16, or NULL (no dgrad copy-back) */
  void *dW;       /* [O, K] bf16 */
} fp8_linear_host_io;
typedef struct {
  void *X, *dY, *Y, *dX, *dW; /* device buffers of the slot (dX may be NULL: no dgrad) */
  void *ctx;                  /* fp8_linear_ctx_size bytes */
  void *ws;                   /* fp8_linear_workspace_size bytes */
  size_t ws_bytes;
} fp8_linear_device_io;
fp8_status fp8_host_pipeline_create(int slots, fp8_host_pipeline **out);
void fp8_host_pipeline_destroy(fp8_host_pipeline *p);
fp8_status fp8_linear_step_host(fp8_host_pipeline *p, int slot, int64_t N,
                                const fp8_linear_host_io *host, const fp8_linear_device_io *dev,
                                fp8_weight_cache *cache, fp8_weight_handle h, fp8_recipe recipe,
                                uint64_t w_version);
fp8_status fp8_host_pipeline_fork(fp8_host_pipeline *p, fp8_stream_t s);
fp8_status fp8_host_pipeline_join(fp8_host_pipeline *p, fp8_stream_t s);
fp8_status fp8_host_pipeline_sync(fp8_host_pipeline *p);

/* ------------------------------------------------------------------ kernel timing
 * Per-kernel timing for roofline reports.  Between fp8_profile_begin and
 * fp8_profile_end every kernel this library launches is bracketed by two
 * CUDA events recorded on its own launch stream, and the launcher's
 * algorithmic byte and flop counts and the problem shape of that launch are
 * recorded with it.  fp8_profile_end synchronises those events and returns
 * one record per kernel name and shape (at most `cap`; *n receives the
 * number of distinct records).  Not thread-safe; host-side bookkeeping only. */
typedef struct {
  char name[64];
  uint64_t launches;
  double total_ms;   /* sum of event-measured durations */
  double bytes;      /* sum of algorithmic HBM bytes (reads + writes) */
  double flops;      /* sum of algorithmic floating-point operations */
  int64_t m, n, k;   /* shape: GEMM M, N, K (split-K reduce: M, N, splits);
                        quantizers rows, cols, 0; elementwise kernels n, 0, 0 */
} fp8_kernel_stat;

fp8_status fp8_profile_begin(void);
fp8_status fp8_profile_end(fp8_kernel_stat *out, int cap, int *n);

/* ------------------------------------------------------------------ allocation-free variant
 * fp8_quantize_tensorwise_noalloc: the tensorwise quantizer of fp8_quantize
 * (recipe FP8_RECIPE_TENSORWISE, same bytes and scales) for callers that
 * cannot allocate device memory, e.g. code running inside a device allocator
 * or memory-pool hook, latency-critical paths that must avoid cudaMalloc /
 * cudaFree (they can synchronise the device), or plugins whose framework owns
 * all device memory.  The reconstruction's pages have no counterpart; this
 * is a library convenience.
 *   The scratch between the two passes (one fp32 partial amax per CTA of the
 *   first pass) lives in a fixed 4 KiB device array inside the library (1024
 *   slots), held on every GPU that loads the library until exit.  The call
 *   needs no workspace and makes no allocation; a launch that would need more
 *   than 1024 slots returns FP8_ERR_WORKSPACE (the first pass uses at most
 *   min(2 x SM count, 1024), so no supported size does).
 *   Every call looks up the array's device address (cudaGetSymbolAddress)
 *   in the current device's context, so a context that was reset and
 *   created again is handled; the first call on a device also loads the
 *   library's device code there, so make that first call before any stream
 *   capture.
 *   All calls on a device share the array and it keeps the last call's
 *   contents; each call overwrites every slot it reads, so nothing needs
 *   clearing.  Calls whose work can overlap on the GPU (unordered streams)
 *   race on the array and must be serialised by the caller.
 *   x [rows, cols] bf16; rowwise_out [rows, cols] and/or colwise_out
 *   [cols, rows] (not both NULL); scale, scale_inv: one float each.
 * Errors: INVALID_ARG, SHAPE, ALIGN, WORKSPACE, CUDA. */
fp8_status fp8_quantize_tensorwise_noalloc(const void *x, int64_t rows, int64_t cols,
                                           fp8_role role, uint8_t *rowwise_out,
                                           uint8_t *colwise_out, float *scale, float *scale_inv,
                                           fp8_stream_t stream);

/* ------------------------------------------------------------------ device status
 * Synchronises `stream`, then returns and clears the device-side status word
 * that kernels set when a bounded wait gives up (FP8_ERR_TIMEOUT) - no kernel
 * traps.  Also returns FP8_ERR_CUDA if the stream reports an error. */
fp8_status fp8_get_device_status(fp8_stream_t stream);

/* Failure-detection test hook: enqueues one kernel that waits, with the same
 * bounded wait the GEMM uses, on a barrier nothing will ever complete; after
 * limit_ns nanoseconds (1 .. 1e9) it records FP8_ERR_TIMEOUT in the device
 * status word and returns (no trap; the context stays usable).  Read the
 * outcome with fp8_get_device_status.  Errors: INVALID_ARG, CUDA. */
fp8_status fp8_debug_wait_timeout(uint64_t limit_ns, fp8_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8LIN_H */
