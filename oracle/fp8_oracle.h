/*
 * fp8_oracle.h -- plain CPU oracle for the per-tensor scaled FP8 linear path.
 *
 * TEST INFRASTRUCTURE ONLY.  This library exists so that the tests, the smoke
 * check and the benchmark's CPU-baseline leg can check the CUDA library against
 * a slow, obviously correct restatement of the method.  The product path never
 * links, loads or calls it, and it shares no source with the CUDA library.
 *
 * Sources (web pages on FP8 mixed precision):
 *   [TE]  "4.2 Hopper I -- Transformer Engine / FP8" (aegloslab.com/nvidia/43):
 *         S4.2.3 the two formats, S4.2.4 amax-based per-tensor scale, scaled cast,
 *         FP32-accumulated GEMM with x(1/scale) dequant, delayed scaling with an
 *         amax history; S4.2.5 worked example; S4.2.6 recipe (history length 16,
 *         "max" rule, HYBRID = E4M3 forward / E5M2 backward); S4.2.8 names the
 *         OCP FP8 standard for the bit layouts.
 *   [LP]  "FP8 and low-precision formats" (aiunderstanding.org), technical-insight
 *         section: scale into the FP8 window, multiply-accumulate, scale back,
 *         partial sums kept in FP16/FP32; format overview: per-block scale
 *         factors and the MX formats; use cases: E5M2 gradient communication.
 *   [FL]  "[📪정보] 그저께 나온 논문 대박이네" (mir.rootios.com, thesingularity board),
 *         a thread on the FP8-LM paper: precision decoupling and automatic
 *         scaling of gradients during the all-reduce.
 *
 * Precision: values are carried in fp64 wherever the pages leave the precision
 * open; the scaled product x*scale and the scale itself are fp32 because the
 * method defines them on fp32 tensors (see each function).
 */
#ifndef FP8_ORACLE_H
#define FP8_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_E4M3 = 0, ORACLE_E5M2 = 1 };

/* Decode one FP8 code to its exact value (NaN / +-Inf as IEEE doubles). */
double oracle_fp8_decode(uint8_t code, int fmt);
/* Largest finite value of the format (448 for E4M3, 57344 for E5M2). */
double oracle_fp8_max(int fmt);
/* Saturating round-to-nearest-even encode of an fp32 value. */
uint8_t oracle_fp8_encode(float v, int fmt);
/* The same for any double (the exact value being rounded). */
uint8_t oracle_fp8_encode_double(double v, int fmt);
/* Element-wise versions over arrays. */
void oracle_fp8_decode_array(const uint8_t* codes, int64_t n, int fmt, double* out);
void oracle_fp8_encode_array(const float* v, int64_t n, int fmt, uint8_t* out);

/* bf16 <-> wider types. */
float oracle_bf16_to_float(uint16_t b);
uint16_t oracle_double_to_bf16(double y);
void oracle_double_to_bf16_array(const double* y, int64_t n, uint16_t* out);

/* amax = max_i |x_i| of a bf16 tensor, as an fp32 value.  NaN dominates. */
float oracle_amax_bf16(const uint16_t* x, int64_t n);

/* Scaled cast q_i = encode(fp32(x_i) * scale); counts saturated and underflowed
 * elements.  Returns nothing; counts go to *n_sat and *n_und. */
void oracle_cast_bf16(const uint16_t* x, int64_t n, float scale, int fmt, uint8_t* q,
                      uint64_t* n_sat, uint64_t* n_und);

/* scale = FP8_MAX / m in fp32 (the previous scale is kept when m is zero or not
 * finite; an overflowing quotient is clamped to FLT_MAX). */
float oracle_scale_from_amax(float m, int fmt, float prev_scale);
/* 1 / scale in fp32. */
float oracle_reciprocal(float s);

/* D rows of the dequantised FP8 GEMM D = (A . B^T) * factor:
 *   A: codes [M, K] row-major (leading dim lda), format afmt
 *   B: codes [N, K] row-major (leading dim ldb), format bfmt
 *   rows: nrows row indices of D to compute (all rows when rows == NULL, nrows = M)
 * For each requested row r (output row i) and every n < N:
 *   acc[i*N+n]  = sum_k dec(A[r,k]) * dec(B[n,k])          (fp64)
 *   absacc[...] = sum_k |dec(A[r,k]) * dec(B[n,k])|        (fp64, error-bound weight)
 *   out[...]    = bf16_rne(acc * (double)factor)            (may be NULL)
 * factor is the fp32 product sinv_a * sinv_b. */
void oracle_gemm_rows(const uint8_t* A, int afmt, int64_t lda, const uint8_t* B, int bfmt,
                      int64_t ldb, int64_t M, int64_t N, int64_t K, const int64_t* rows,
                      int64_t nrows, float factor, double* acc, double* absacc, uint16_t* out);

/* Block scaling, MX style ([LP]: per-block scale factors, MXFP8).  A block is 32
 * consecutive elements of a row (the row's last block may be shorter); its scale
 * is 2^-k, stored as the E8M0 code 127 - k, with k the largest integer in
 * [-127, 127] such that amax_block * 2^k <= FP8_MAX (-127 if none: Inf/NaN).
 * Elements: q = round_to_fp8(x * 2^k) (exact product, saturating RNE). */
int oracle_mx_scale_exponent(double amax, int fmt);
/* Value of an E8M0 scale code: 2^(code-127); 0xFF is NaN. */
double oracle_e8m0_value(uint8_t code);
/* x: bf16 [rows, cols] row-major; q: codes [rows, cols]; scale: E8M0 codes
 * [rows, ceil(cols/32)] row-major. */
void oracle_mx_quantize(const uint16_t* x, int64_t rows, int64_t cols, int fmt, uint8_t* q,
                        uint8_t* scale);
/* Rows of D = dequant(A) . dequant(B)^T with A [M, K], B [N, K] codes (contiguous
 * rows) and their E8M0 block scales sa [M, ceil(K/32)], sb [N, ceil(K/32)]:
 *   acc    = sum_k (dec(A[r,k]) * 2^(sa-127)) * (dec(B[n,k]) * 2^(sb-127))   (fp64)
 *   absacc = the same sum of magnitudes; out = bf16_rne(acc) (may be NULL). */
void oracle_mx_gemm_rows(const uint8_t* A, int afmt, const uint8_t* sa, const uint8_t* B, int bfmt,
                         const uint8_t* sb, int64_t M, int64_t N, int64_t K, const int64_t* rows,
                         int64_t nrows, double* acc, double* absacc, uint16_t* out);

/* FP8 (E5M2) gradient all-reduce with automatic scaling ([LP] use cases; [FL]
 * forum thread on the FP8-LM paper: "automatic scaling").  g: bf16 [world][n],
 * rank r's gradient at g + r*n.  Shared scale s = 57344 / fp32(world * amax)
 * (amax over all ranks; 1 for a zero or non-finite amax; FLT_MAX clamps); each
 * rank's codes are E5M2(fp32(g*s)); their exact sum is rounded to E5M2 (the
 * reduced code, into `codes` if not NULL); out = bf16(fp32(decode(code) * f)),
 * f = 1/s, or fp32((1/s)/world) when `average`.  scale (may be NULL) gets
 * {s, 1/s}. */
float oracle_allreduce_scale(float amax, int world);
void oracle_allreduce_e5m2(const uint16_t* g, int world, int64_t n, int average, uint16_t* out,
                           uint8_t* codes, float* scale);

/* The next stage's cast composed into a GEMM epilogue ([TE] S4.2.4: the FP32
 * result is multiplied by 1/scale "or composed with the next stage's scale"):
 * v holds the fp32 values the epilogue stores, q_i = encode(fp32(v_i * scale)).
 * Counts as oracle_cast_bf16: saturated |fp32(v*scale)| > FP8_MAX, underflowed
 * v != 0 with a +-0 code; *amax = max |v| (NaN dominates). */
void oracle_cast_f32(const float* v, int64_t n, float scale, int fmt, uint8_t* q, uint64_t* n_sat,
                     uint64_t* n_und, float* amax);

/* The activation between FC1 and FC2 of the transformer layer's MLP ([TE]
 * S4.2.6 builds its model from te.TransformerLayer; the page does not name
 * the function -- reading: GELU in its tanh form), in fp64:
 *   gelu(x)  = x/2 * (1 + tanh(c * (x + 0.044715 x^3))),  c = sqrt(2/pi)
 *   dgelu(x) = d gelu / dx. */
double oracle_gelu(double x);
double oracle_dgelu(double x);
void oracle_gelu_array(const double* x, int64_t n, double* out);
void oracle_dgelu_array(const double* x, int64_t n, double* out);

/* Number of OpenMP threads the oracle runs with. */
int oracle_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
