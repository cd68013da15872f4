/*
 * fp8lin.h -- C ABI of libfp8lin: the per-tensor, dynamically scaled FP8 linear
 * layer on one GB300 (sm_103a).
 *
 * The method ("4.2 Hopper I -- Transformer Engine / FP8", aegloslab.com/nvidia/43):
 *   S4.2.3  two 8-bit formats: E4M3 (weights, activations) and E5M2 (gradients);
 *           exact layouts per OCP FP8, the standard S4.2.8 names.
 *   S4.2.4  per tensor: amax = max|x|, scale = FP8_MAX / amax,
 *           x_fp8 = round_to_fp8(x * scale); the GEMM runs on FP8 inputs,
 *           accumulates in FP32 and multiplies by 1/scale of each operand.
 *           Delayed scaling: the scale comes from a history of past amaxes
 *           (max of the last N), so the cast needs one pass over the tensor.
 *   S4.2.6  recipe: HYBRID format (E4M3 forward, E5M2 backward),
 *           amax_history_len = 16, amax_compute_algo = "max"; the library
 *           updates the amaxes to set the next step's scales.
 * ("FP8 and low-precision formats", aiunderstanding.org, technical insight:
 *  scale into the FP8 window, multiply-accumulate, scale back, accumulate
 *  partial sums in FP16/FP32.)
 *
 * Conventions for every call:
 *  - Tensor buffers are DEVICE pointers owned by the caller; the library never
 *    frees or retains them past the call's stream work.
 *  - Matrices are row-major.  bf16 inputs are IEEE bfloat16 bit patterns; FP8
 *    outputs are one byte per element (OCP E4M3 or E5M2 codes).
 *  - Calls enqueue work on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and return without synchronising, except fp8_get_state,
 *    fp8_set_state, fp8_check_device_error and fp8_recipe_destroy.
 *  - Errors: every call returns an fp8_status_t.  Argument errors are found on
 *    the host before anything is enqueued (FP8_ERR_INVALID / _UNSUPPORTED);
 *    CUDA launch/runtime errors give FP8_ERR_CUDA.  Kernels never trap: a device
 *    wait that exceeds its time limit records an error word in the recipe and
 *    returns; the next synchronising call reports FP8_ERR_TIMEOUT.
 *    fp8_last_error_message() gives the calling thread's last detail string.
 *  - Calls on one recipe that run concurrently on different streams and touch
 *    the same tensor id race; order them on one stream.  GEMMs on one recipe
 *    must not overlap at all (they share its split-tail workspace).
 *  - The casts, the scale update and the GEMMs are launched with programmatic
 *    dependent launch: a kernel may start while the previous kernel on the
 *    stream finishes, but waits for it to complete before it reads or writes
 *    any memory, so stream order holds as for plain launches (also under CUDA
 *    graph capture).  Setting FP8LIN_PDL=0 in the environment launches them
 *    plainly.
 */
#ifndef FP8LIN_H
#define FP8LIN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct fp8_recipe fp8_recipe_t; /* opaque; owned by the library */
typedef void* fp8_stream_t;             /* a cudaStream_t */

typedef enum {
  FP8_OK = 0,
  FP8_ERR_INVALID = 1,     /* bad argument (null, size, alignment, id, enum) */
  FP8_ERR_UNSUPPORTED = 2, /* valid request the library does not implement */
  FP8_ERR_CUDA = 3,        /* CUDA runtime / driver error */
  FP8_ERR_TIMEOUT = 4,     /* a device-side wait ran past its limit */
  FP8_ERR_NOMEM = 5        /* device or host allocation failed */
} fp8_status_t;

typedef enum { FP8_E4M3 = 0, FP8_E5M2 = 1 } fp8_dtype_t;
typedef enum { FP8_RECIPE_HYBRID = 0, FP8_RECIPE_E4M3 = 1 } fp8_recipe_format_t;
typedef enum { FP8_AMAX_MAX = 0, FP8_AMAX_MOST_RECENT = 1 } fp8_amax_algo_t;
typedef enum { FP8_SCALING_DELAYED = 0, FP8_SCALING_CURRENT = 1 } fp8_scaling_t;
/* GEMM output: bf16 or fp32 values of the dequantised product, or FP8 codes of
 * that product times the output tensor's scale (the next stage's scale
 * composed into the epilogue, S4.2.4). */
typedef enum { FP8_OUT_BF16 = 0, FP8_OUT_F32 = 1, FP8_OUT_E4M3 = 2, FP8_OUT_E5M2 = 3 } fp8_out_dtype_t;
/* Storage of a GEMM operand: K-major = [M or N rows, K] (K contiguous);
 * MN-major = [K rows, M or N] (M or N contiguous). */
typedef enum { FP8_K_MAJOR = 0, FP8_MN_MAJOR = 1 } fp8_major_t;

/* Snapshot of one tensor's scaling state (fp8_get_state). */
typedef struct {
  float scale;             /* scale the next DELAYED cast of this tensor uses */
  float scale_inv;         /* 1/scale, fp32 round-to-nearest */
  float cast_scale;        /* scale the most recent cast used */
  float cast_scale_inv;    /* its reciprocal: the GEMM dequantises with this */
  float amax_pending;      /* max |x| recorded since the last history update */
  float amax_last;         /* amax the most recent history update pushed */
  uint64_t n_saturated;    /* #elements with |x*scale| > FP8_MAX since the last update */
  uint64_t n_underflow;    /* #nonzero elements cast to +-0 since the last update */
  uint64_t n_saturated_last; /* the two counts the most recent update closed */
  uint64_t n_underflow_last;
  int32_t dtype;           /* fp8_dtype_t of the most recent cast (sets FP8_MAX) */
  int32_t recorded;        /* 1 if an amax was recorded since the last update */
} fp8_tensor_state_t;

/* Create a scaling recipe for `num_tensors` tensors (ids 0..num_tensors-1),
 * each with an amax history of `amax_history_len` (S4.2.6 uses 16) reduced by
 * `algo` (S4.2.6 uses "max").  `format` HYBRID allows E4M3 and E5M2 casts;
 * E4M3 rejects E5M2 casts.  Initial state of every tensor: history all 0,
 * scale = scale_inv = cast_scale = cast_scale_inv = 1, nothing recorded.
 * Allocates device state (enqueued on `stream`, which is synchronised): the
 * tensors' states and histories, and the GEMMs' split-tail workspace (256 KB
 * per pair of SMs, about 19 MB on a 152-SM GPU).
 * Errors: INVALID (null out, history_len < 1 or > 1024, num_tensors < 1 or
 * > 65536, unknown enum), NOMEM, CUDA. */
fp8_status_t fp8_recipe_create(fp8_recipe_t** out, int32_t format, int32_t amax_history_len,
                               int32_t algo, int32_t num_tensors, fp8_stream_t stream);

/* Synchronise the device and free the recipe's device state.  NULL is a no-op. */
fp8_status_t fp8_recipe_destroy(fp8_recipe_t* r);

/* amax + scale + saturating cast of one bf16 tensor (S4.2.4).
 *   x:      bf16 [rows, cols] row-major, 16-byte aligned (n = rows*cols >= 1).
 *   dtype:  FP8_E4M3 (FP8_MAX 448) or FP8_E5M2 (FP8_MAX 57344).
 *   mode:   DELAYED -- cast with the tensor's current `scale` (from its history)
 *           in ONE pass that also records amax(x);
 *           CURRENT -- first measure amax(x), then cast with
 *           scale = FP8_MAX/amax(x) (two passes; S4.2.4 calls this the slow way).
 *   out:    n bytes, FP8 codes of x*scale, same layout as x, 16-byte aligned.
 *   out_t:  NULL, or cols*rows bytes receiving the transposed codes [cols, rows],
 *           16-byte aligned: K-major operands for the backward GEMMs of the
 *           Hopper layout.  fp8_gemm_layout reads `out` MN-major instead, so
 *           the backward GEMMs need no transposed copy.
 *   update_now: nonzero = after the cast, push this tensor's pending amax into
 *           its history and recompute scale/scale_inv at once (a one-thread
 *           launch on the same stream); zero = leave that to fp8_update_scales.
 * Per cast, the tensor's state records: amax into amax_pending (max with what
 * the step already holds), saturated / underflowed counts, cast_scale and
 * cast_scale_inv, dtype.  Errors: INVALID (null/unaligned pointers, n < 1,
 * bad id/enum, E5M2 on an E4M3 recipe), CUDA. */
fp8_status_t fp8_amax_quantize(fp8_recipe_t* r, int32_t tensor_id, const void* x, int64_t rows,
                               int64_t cols, int32_t dtype, int32_t mode, int32_t update_now,
                               void* out, void* out_t, fp8_stream_t stream);

/* Dequantised FP8 GEMM on the tensor cores (S4.2.4):
 *   y[m, n] = ( sum_k A[m, k] * B[n, k] ) * (cast_scale_inv[a_id] * cast_scale_inv[b_id])
 * with FP32 accumulation; the product of the two reciprocal scales is an fp32
 * multiply; D = y as bf16 (round-to-nearest-even) or fp32 -- or, with d_dtype
 * FP8_OUT_E4M3 / FP8_OUT_E5M2, D = round_to_fp8(y * scale[amax_out_id]) with
 * saturation: the result's 1/scale composed with the next stage's scale
 * (S4.2.4), the output tensor's delayed scale.  Then that tensor's state
 * records max|y| (into amax_pending), the saturated / underflowed counts,
 * cast_scale = its scale, cast_scale_inv = its scale_inv and the dtype, as a
 * delayed-scaling cast of y would.
 *   A: FP8 codes [M, K] row-major (K contiguous), row stride lda bytes.
 *   B: FP8 codes [N, K] row-major (K contiguous), row stride ldb bytes.
 *      Forward Y = X W^T: A = Xq [T, in], B = Wq [out, in].
 *      dgrad dX = dY W:   A = dYq [T, out], B = Wq^T [in, out] (out_t of W).
 *      wgrad dW = dY^T X: A = dYq^T [out, T], B = Xq^T [in, T] (out_t of dY, X).
 *      (fp8_gemm_layout runs both on the untransposed codes.)
 *   a_dtype, b_dtype: FP8_E4M3 / FP8_E5M2, any combination.
 *   D: [M, N] row-major with row stride ldd elements of d_dtype (bytes for
 *           the FP8 outputs).
 *   amax_out_id: -1, or a tensor id whose amax_pending takes max|D| of the
 *           stored values (the next layer's amax, fused into the epilogue);
 *           required for FP8 outputs (max|y| before the output scale).
 * Requirements: M, N >= 1; K >= 16 and K % 16 == 0; lda, ldb >= K and
 * multiples of 16; A, B 16-byte aligned; ldd >= N.  Errors: INVALID (also: an
 * FP8 output without amax_out_id, an E5M2 output on an E4M3 recipe), CUDA.
 * GEMMs on one recipe must run one after another on the device (one stream,
 * or streams ordered by events): the last, partial wave of output tiles is
 * shared out across the GPU through a workspace that the recipe owns (one
 * 256 KB slot per pair of SMs, allocated by fp8_recipe_create).  The result
 * does not depend on the stream or on other launches. */
fp8_status_t fp8_gemm(fp8_recipe_t* r, int32_t a_id, const void* A, int32_t a_dtype, int64_t lda,
                      int32_t b_id, const void* B, int32_t b_dtype, int64_t ldb, int64_t M,
                      int64_t N, int64_t K, void* D, int32_t d_dtype, int64_t ldd,
                      int32_t amax_out_id, fp8_stream_t stream);

/* fp8_gemm with each operand's storage chosen (the same product, epilogue,
 * state updates and errors):
 *   a_major: FP8_K_MAJOR -- A is [M, K], row stride lda >= K;
 *            FP8_MN_MAJOR -- A is stored [K, M] (element (m, k) at k*lda + m),
 *            lda >= M.
 *   b_major: FP8_K_MAJOR -- B is [N, K], ldb >= K;
 *            FP8_MN_MAJOR -- B is stored [K, N] (element (n, k) at k*ldb + n),
 *            ldb >= N.
 * The tensor cores read either layout, so the backward GEMMs can use the
 * forward casts' codes without transposed copies (S4.2.4's three GEMMs):
 *   dgrad dX = dY W:   A = dYq [T, out] K-major, B = Wq [out, in] MN-major;
 *   wgrad dW = dY^T X: A = dYq [T, out] MN-major, B = Xq [T, in] MN-major.
 * lda, ldb: multiples of 16.  Both kernel variants (FP8LIN_GEMM_KERNEL unset
 * or "one") read either layout.
 * Errors: as fp8_gemm; INVALID also for an unknown layout. */
fp8_status_t fp8_gemm_layout(fp8_recipe_t* r, int32_t a_id, const void* A, int32_t a_dtype, int32_t a_major,
                             int64_t lda, int32_t b_id, const void* B, int32_t b_dtype, int32_t b_major,
                             int64_t ldb, int64_t M, int64_t N, int64_t K, void* D, int32_t d_dtype,
                             int64_t ldd, int32_t amax_out_id, fp8_stream_t stream);

/* Activation fused into the GEMM epilogue: the glue between the two GEMMs of
 * the transformer layer's MLP (S4.2.6 builds its model from
 * te.TransformerLayer, hidden 4096, FFN 16384: FC1 -> activation -> FC2).
 * The pages do not name the function; it is GELU in its tanh form,
 *   gelu(x)  = x/2 * (1 + t),  t = tanh(c * (x + a * x^3)),  c = sqrt(2/pi), a = 0.044715,
 *   gelu'(x) = (1 + t)/2 + x/2 * (1 - t^2) * c * (1 + 3a * x^2),
 * evaluated in fp32 on the dequantised result y (the same fp32 value whatever
 * the output type), with (1 + t)/2 computed as 1 / (1 + e^(-2u)) through the
 * fast exponential and reciprocal (relative error a few 1e-7 times
 * (1 + |2u|); far below the spacing of the FP8 codes the chained step stores). */
typedef enum { FP8_ACT_NONE = 0, FP8_ACT_GELU = 1, FP8_ACT_DGELU = 2 } fp8_act_t;

/* fp8_gemm_layout with an activation between the dequantised product and the
 * store, so that a GEMM can write the next GEMM's FP8 operand (S4.2.4: the
 * result is multiplied by 1/scale "or composed with the next stage's scale"):
 *   FP8_ACT_NONE:  exactly fp8_gemm_layout; aux must be NULL.
 *   FP8_ACT_GELU:  the stored value is gelu(y); aux, when not NULL, receives
 *                  bf16(gelu'(y)) -- the derivative the backward multiplies
 *                  by (computed from the same exponential as gelu(y)).  The
 *                  forward FC1 GEMM: D = FC2's input X, e.g. as E4M3 codes
 *                  with amax_out_id = FC2's X tensor.
 *   FP8_ACT_DGELU: the stored value is y * aux, aux (required) = the
 *                  forward's bf16 gelu'(y): FC2's dgrad, D = FC1's output
 *                  gradient, e.g. as E5M2 codes with amax_out_id = FC1's dY
 *                  tensor.
 * D, d_dtype and amax_out_id act on the stored value as in fp8_gemm (an FP8
 * output records max|value|, the counts of its cast and the cast's scale).
 *   aux: bf16 [M, N], row stride ld_aux elements (caller's buffer): 16-byte
 *        aligned, ld_aux >= N, ld_aux % 8 == 0 and N % 8 == 0.
 * Errors: as fp8_gemm_layout; INVALID also for an unknown activation, a
 * missing or misaligned aux, or an aux without an activation. */
fp8_status_t fp8_gemm_act(fp8_recipe_t* r, int32_t a_id, const void* A, int32_t a_dtype, int32_t a_major,
                          int64_t lda, int32_t b_id, const void* B, int32_t b_dtype, int32_t b_major, int64_t ldb,
                          int64_t M, int64_t N, int64_t K, void* D, int32_t d_dtype, int64_t ldd,
                          int32_t amax_out_id, int32_t act, void* aux, int64_t ld_aux, fp8_stream_t stream);

/* End of step (S4.2.6): for every tensor that recorded an amax since the last
 * update, push amax_pending into its history (dropping the oldest entry), set
 * scale = FP8_MAX(dtype) / reduce(history) in fp32 (reduce = max or newest
 * entry) and scale_inv = 1/scale, move the step's counts to *_last and reset
 * them.  A zero or non-finite reduced amax keeps the previous scale; an
 * overflowing quotient is clamped to FLT_MAX.  One kernel launch. */
fp8_status_t fp8_update_scales(fp8_recipe_t* r, fp8_stream_t stream);

/* Copy one tensor's state to the host (synchronises `stream`).  `history` may
 * be NULL, else receives amax_history_len floats, oldest first.  Returns
 * FP8_ERR_TIMEOUT if a kernel on this recipe recorded a device timeout. */
fp8_status_t fp8_get_state(fp8_recipe_t* r, int32_t tensor_id, fp8_tensor_state_t* state,
                           float* history, fp8_stream_t stream);

/* Overwrite one tensor's history (amax_history_len floats, oldest first, each
 * >= 0) and scale (finite, > 0); sets scale_inv = cast_scale_inv = 1/scale,
 * cast_scale = scale, the dtype, and clears pending amax and counts.
 * Synchronises `stream`.  Used for warm starts and checkpoint/resume. */
fp8_status_t fp8_set_state(fp8_recipe_t* r, int32_t tensor_id, const float* history, float scale,
                           int32_t dtype, fp8_stream_t stream);

/* Synchronise `stream` and report (then clear) a device-side timeout recorded
 * by any kernel of this recipe: FP8_OK or FP8_ERR_TIMEOUT. */
fp8_status_t fp8_check_device_error(fp8_recipe_t* r, fp8_stream_t stream);

/* ---- MX block scaling --------------------------------------------------------
 * "FP8 and low-precision formats" (aiunderstanding.org), format overview:
 * scale factors per tensor OR PER BLOCK; the MX formats (MXFP8 among them)
 * share one scale per small block of elements.  The page gives no rule; this
 * library reads the block scale as the per-tensor rule of S4.2.4 above
 * (FP8_MAX / amax) restricted to powers of two:
 *   block: 32 consecutive elements of a row (a row's last block may hold 16);
 *   k:     the largest integer in [-127, 127] with amax_block * 2^k <= FP8_MAX,
 *          -127 when there is none (an Inf or NaN in the block);
 *   scale: one E8M0 byte 127 - k = the block's dequantisation factor 2^-k;
 *   q:     round_to_fp8(x * 2^k), saturating round-to-nearest-even.
 * No recipe state is read or written: the scales travel with the codes.  The
 * recipe argument only supplies the device error word for time-outs.
 *
 * Scale layout ("atoms"): the scales of a [rows, cols] matrix are
 * ceil(rows/128) x ceil(cols/128) atoms of 512 bytes, row-major by atom.  The
 * scale of row r, block b (columns 32b..32b+31) is at byte
 *     ((r / 128) * ceil(cols / 128) + b / 4) * 512
 *       + (r % 32) * 16 + ((r / 32) % 4) * 4 + (b % 4)
 * -- the order in which the tensor cores' block-scaled MMA reads scales from
 * tensor memory after one 512-byte copy per 128 rows x 128 columns.  Entries of
 * rows >= rows or blocks >= ceil(cols/32) are padding: fp8_mx_quantize writes 0
 * there, and fp8_mx_gemm needs them finite (any code but 0xFF). */

/* Bytes of the scale array of a [rows, cols] MX matrix; -1 for sizes < 1. */
int64_t fp8_mx_scale_bytes(int64_t rows, int64_t cols);

/* MX quantisation of a bf16 matrix (one kernel, one read of x):
 *   x:         bf16 [rows, cols] row-major, contiguous, 16-byte aligned.
 *   dtype:     FP8_E4M3 or FP8_E5M2 (FP8_MAX 448 / 57344).
 *   q:         rows*cols bytes: codes of x, blocks along each row.
 *   q_scale:   fp8_mx_scale_bytes(rows, cols) bytes: their scales (atoms).
 *   q_t:       NULL, or cols*rows bytes: codes of x^T [cols, rows] quantised
 *              with ITS OWN blocks (32 consecutive rows of x), the K-major
 *              operand the backward GEMMs need -- not a transpose of q.
 *   q_t_scale: NULL with q_t, else fp8_mx_scale_bytes(cols, rows) bytes.
 * Requirements: 1 <= rows <= 2^30; cols a multiple of 16 in [16, 2^30];
 * rows % 16 == 0 when q_t is given; every pointer 16-byte aligned.  All
 * buffers are the caller's.  Errors: INVALID, CUDA; a device time-out shows at
 * the next synchronising call of the recipe (FP8_ERR_TIMEOUT). */
fp8_status_t fp8_mx_quantize(fp8_recipe_t* r, const void* x, int64_t rows, int64_t cols, int32_t dtype,
                             void* q, void* q_scale, void* q_t, void* q_t_scale, fp8_stream_t stream);

/* Block-scaled FP8 GEMM on the tensor cores:
 *   D[m, n] = sum_k (A[m,k] * 2^-ka(m, k/32)) * (B[n,k] * 2^-kb(n, k/32))
 * with the products' block sums accumulated in FP32 (partial sums promoted
 * into round-to-nearest FP32 every 2048 of K), D stored as bf16 (RNE) or fp32.
 *   A: FP8 codes [M, K] (K contiguous, row stride lda bytes), a_scale its
 *      scales in the atom layout of an [M, K] matrix.
 *   B: FP8 codes [N, K] (row stride ldb bytes), b_scale those of [N, K].
 *      Forward Y = X W^T: A = q(X), B = q(W); dgrad dX = dY W: A = q(dY),
 *      B = q_t(W); wgrad dW = dY^T X: A = q_t(dY), B = q_t(X).
 *   a_dtype, b_dtype: FP8_E4M3 / FP8_E5M2, any combination.
 *   D: [M, N] row-major, row stride ldd elements; d_dtype FP8_OUT_BF16 or
 *      FP8_OUT_F32.
 * Requirements: M, N >= 1; K >= 16 and K % 16 == 0; lda, ldb >= K and
 * multiples of 16; A, B, a_scale, b_scale 16-byte aligned; ldd >= N.
 * Errors: INVALID, CUDA; device time-outs as for fp8_mx_quantize. */
fp8_status_t fp8_mx_gemm(fp8_recipe_t* r, const void* A, int32_t a_dtype, int64_t lda, const void* a_scale,
                         const void* B, int32_t b_dtype, int64_t ldb, const void* b_scale, int64_t M,
                         int64_t N, int64_t K, void* D, int32_t d_dtype, int64_t ldd, fp8_stream_t stream);

/* ---- FP8 (E5M2) gradient all-reduce with automatic scaling --------------------
 * "FP8 and low-precision formats" (aiunderstanding.org), use cases: E5M2 for
 * gradient communication in distributed training, to cut inter-node
 * bandwidth.  "[📪정보] 그저께 나온 논문 대박이네" (mir.rootios.com, a thread on the
 * FP8-LM paper): automatic scaling of the tensor scaling factor keeps the
 * gradients inside FP8's range during the all-reduce.  These four calls are
 * the device steps; the exchange between ranks (a MAX all-reduce of one float,
 * an all-to-all and an all-gather of bytes) is the caller's, e.g. through
 * torch.distributed:
 *   1. fp8_grad_amax        local amax -> MAX across ranks -> shared amax
 *   2. fp8_grad_quantize    codes = E5M2(fp32(g * s)), s = 57344 / fp32(world * amax)
 *   3. all-to-all           rank r receives chunk r of every rank: [world][chunk]
 *   4. fp8_grad_reduce      exact sum of the world codes, rounded to E5M2
 *   5. all-gather           of the reduced chunks: [world * chunk]
 *   6. fp8_grad_dequantize  bf16(fp32(decode(code) * f)), f = 1/s or (1/s)/world
 * No recipe is involved; none of the kernels waits, so none can time out.
 * Inputs are bf16; a NaN input makes a NaN result (its byte codes are not
 * specified further). */
#define FP8_GRAD_MAX_WORLD 32768

/* max|g| of a bf16 vector into *amax (device float; NaN dominates).  The call
 * zeroes *amax first on the same stream.  g: n >= 1 elements, 16-byte aligned. */
fp8_status_t fp8_grad_amax(const void* g, int64_t n, float* amax, fp8_stream_t stream);

/* codes[i] = E5M2(fp32(g[i] * s)) for i < n and 0 for n <= i < padded_n, with
 * the shared scale s = 57344 / fp32(world * amax[0]) (world * amax clamped to
 * FLT_MAX; s = 1 when amax is 0 or not finite; s clamped to FLT_MAX).
 * scale (2 device floats) receives {s, 1/s}.  g, codes 16-byte aligned;
 * 1 <= world <= FP8_GRAD_MAX_WORLD; padded_n >= n. */
fp8_status_t fp8_grad_quantize(const void* g, int64_t n, const float* amax, int32_t world, void* codes,
                               int64_t padded_n, float* scale, fp8_stream_t stream);

/* out[i] = E5M2(sum over r < world of decode(recv[r * chunk + i])), i < chunk:
 * the sum is exact (multiples of 2^-16: two fp32 values per element up to 128
 * ranks, 64-bit integers above) and rounded once, to nearest with ties to the
 * even code, saturating at 57344; a sum of negative zeros is -0; an Inf or
 * NaN code among the addends gives the NaN code 0x7E.  recv [world][chunk],
 * out [chunk], 16-byte aligned; chunk a positive multiple of 16. */
fp8_status_t fp8_grad_reduce(const void* recv, int32_t world, int64_t chunk, void* out, fp8_stream_t stream);

/* out[i] = bf16(fp32(decode(codes[i]) * f)) for i < n, f = scale[1] (the sum)
 * or fp32(scale[1] / world) when average != 0 (the mean).  codes and out
 * 16-byte aligned; out is bf16 [n]. */
fp8_status_t fp8_grad_dequantize(const void* codes, int64_t n, const float* scale, int32_t world,
                                 int32_t average, void* out, fp8_stream_t stream);

/* Largest n fp8_quantize_current_noalloc accepts: 16384 blocks of 65536
 * elements, the per-block slots of its static scratch (192 KiB per GPU). */
#define FP8_NOALLOC_MAX_ELEMENTS ((int64_t)1 << 30)

/* Current-scaling cast that allocates nothing.  The pages have no counterpart:
 * this entry point exists for callers that cannot call cudaMalloc -- code that
 * runs inside a host framework which owns all device memory and forbids
 * allocation while it executes (a plugin's enqueue step, a fixed memory plan),
 * or code that must not risk the device-wide synchronisation an allocation can
 * cause.  It needs no recipe.
 *   x:          bf16 [n] device pointer, 16-byte aligned, 1 <= n <= FP8_NOALLOC_MAX_ELEMENTS.
 *   dtype:      FP8_E4M3 or FP8_E5M2.
 *   out:        n bytes (device, 16-byte aligned): codes of x*scale, where
 *               scale = FP8_MAX/amax(x) in fp32 (1 when amax is 0 or not finite,
 *               FLT_MAX when the quotient overflows) -- the same codes, scale and
 *               counts as fp8_amax_quantize in CURRENT mode on a fresh recipe.
 *   scale_out:  2 floats (device): {scale, 1/scale}.
 *   counts_out: NULL or 2 uint64 (device): {#saturated, #underflowed}.
 * Scratch: a file-scope __device__ array of the library (one per GPU that loads
 * it, kept until the process exits).  The first call on a device looks up its
 * device address (cudaGetSymbolAddress) and keeps it for the rest of the
 * process; make that first call before any stream capture.  The kept address
 * belongs to the device's primary context: it is not looked up again after
 * cudaDeviceReset, so do not call this entry point after resetting a device.  Every call clears the array's two counters with
 * cudaMemsetAsync and otherwise overwrites what it reads, so the array keeps
 * only the last call's contents; calls that overlap on the GPU (on unordered
 * streams) race on it.  No cudaMalloc/cudaFree or allocating library routine is
 * called.  Errors: INVALID (null or unaligned pointer, unknown dtype, n outside
 * [1, FP8_NOALLOC_MAX_ELEMENTS]), CUDA. */
fp8_status_t fp8_quantize_current_noalloc(const void* x, int64_t n, int32_t dtype, void* out,
                                          float* scale_out, uint64_t* counts_out,
                                          fp8_stream_t stream);

/* ---- failure detection test hook ---------------------------------------------
 * Every device wait of the library is bounded (about 1 s in the casts, 2 s in
 * the GEMMs); a wait that runs out records an error bit in the recipe and the
 * kernel returns -- the next synchronising call reports FP8_ERR_TIMEOUT and the
 * CUDA context stays usable.  This call makes that happen on purpose, once,
 * for tests: the next launch of the chosen kernel on this recipe over-states
 * its first shared-memory stage's byte count by 16, so that stage's wait can
 * never complete and times out (the copy itself completes normally: nothing is
 * left in flight, nothing faults).
 *   FP8_STALL_CAST: the next fp8_amax_quantize with a transposed copy and
 *                   cols % 8 == 0 (the kernel that stages tiles by TMA; the
 *                   flat cast has no waits);
 *   FP8_STALL_GEMM: the next fp8_gemm or fp8_gemm_layout (every kernel variant).
 * Errors: INVALID (NULL recipe, unknown target). */
enum { FP8_STALL_CAST = 0, FP8_STALL_GEMM = 1 };
fp8_status_t fp8_debug_inject_stall(fp8_recipe_t* r, int32_t which);

/* Static description of a status code. */
const char* fp8_status_string(fp8_status_t st);

/* Detail of the calling thread's most recent failed call ("" if none). */
const char* fp8_last_error_message(void);

#ifdef __cplusplus
}
#endif
#endif /* FP8LIN_H */
