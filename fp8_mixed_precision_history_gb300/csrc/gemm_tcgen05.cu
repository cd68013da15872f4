// gemm_tcgen05.cu -- dequantised FP8 GEMM on the 5th-generation tensor cores.
//
// "4.2 Hopper I -- Transformer Engine / FP8" (aegloslab.com/nvidia/43), S4.2.4:
// the GEMM runs on FP8 inputs, accumulates in FP32 and multiplies the result by
// 1/scale of each operand.  Here:
//   D[m, n] = bf16_rn( fp32( sum_k A[m,k] * B[n,k] ) * (sinv_A * sinv_B) )
// A [M, K] and B [N, K] are FP8 codes with K contiguous (E4M3 and/or E5M2), or
// either operand MN-major: A stored [K, M], B stored [K, N].  The tensor cores
// read both layouts (the instruction descriptor's major bits); an MN-major
// tile is TMA-loaded as 128 K rows of 128 M or N bytes, B as two such chunks.
// So the backward GEMMs read the forward codes of W, dY and X as they are, and
// the casts write no transposed copies: dgrad dX = dY W takes B = Wq [out, in]
// MN-major; wgrad dW = dY^T X takes A = dYq [T, out] and B = Xq [T, in] MN-major.
//
// Two variants share the design below.
//   fp8_gemm_pair_kernel: a cluster of two CTAs per TPC computes 256x256 tiles
//     with tcgen05.mma.cta_group::2, each CTA holding half of A and half of B,
//     in 256-byte K stages (eight MMAs per stage).  The default for M > 128:
//     its tensor pipe is busy about 92 % of active cycles on the
//     transformer-layer shapes, 16-20 % faster than the one-CTA kernel.
//   fp8_gemm_kernel<OUT, ACT>: one CTA per SM, 128x256 tiles; M <= 128, or
//     FP8LIN_GEMM_KERNEL=one.
// ACT fuses the MLP's activation (GELU, or its derivative in the backward)
// into the epilogue, before the output is cast (act_prepass).
// Design of the one-CTA kernel (sm_103a, persistent over 128x256 output tiles):
//   warp 0      TMA producer: cp.async.bulk.tensor 2-D loads of a 128x128-byte
//               A tile and a 256x128-byte B tile per stage (128-byte swizzle,
//               out-of-range elements zero-filled) into a 4-stage ring.
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 partial-sum
//               buffers) and, from one thread, issues tcgen05.mma.kind::f8f6f4
//               (M=128, N=256, K=32 per instruction, 4 per stage).
//   warps 2..9  epilogue, two warps per TMEM lane quarter (128 columns each).
// Two-level accumulation: the tensor cores' FP8 accumulation into TMEM was
// measured to lose more than round-to-nearest fp32 summation would (its error
// grows with the number of accumulation steps, like truncation).  So every
// kGroup k-blocks (K = 2048) the MMA warp starts a fresh partial sum in the
// other TMEM buffer, and the epilogue warps add each finished partial into fp32
// registers with round-to-nearest (the CUDA-core "promotion" of the pages'
// DeepGEMM discussion, here on TMEM partials).  At the end of a tile the
// registers are multiplied by sinv_A*sinv_B, rounded to bf16 (or kept fp32),
// stored, and optionally folded into a tensor's amax (the next layer's).  The
// two buffers let the epilogue drain one partial while the MMAs fill the other,
// across tile boundaries too.
// Every mbarrier wait is bounded (about 2 s of wall clock); on expiry the CTA
// records an error bit in the recipe, drains its own copies and MMAs (bounded),
// frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "state.cuh"
#include "tc_ptx.cuh"

namespace fp8lin {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;  // bytes = elements
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int ACC = 2;                 // TMEM partial-sum buffers
constexpr int TMEM_COLS = ACC * BN;    // 512
#ifndef FP8LIN_KGROUP
#define FP8LIN_KGROUP 16
#endif
#ifndef FP8LIN_EPI_BATCH
#define FP8LIN_EPI_BATCH 1
#endif
constexpr int kGroup = FP8LIN_KGROUP;  // k-blocks per TMEM partial
constexpr int kEpiBatch = FP8LIN_EPI_BATCH;  // 8-column TMEM loads in flight per wait
constexpr int EPI_WARPS = 8;
constexpr int THREADS = (2 + EPI_WARPS) * 32;
constexpr int EPI_COLS = BN / 2;       // columns per epilogue warp
#ifndef FP8LIN_GROUP_M
#define FP8LIN_GROUP_M 16
#endif
#ifndef FP8LIN_GROUP_M2
#define FP8LIN_GROUP_M2 16
#endif
#ifndef FP8LIN_PAIR_BK
#define FP8LIN_PAIR_BK 256
#endif
#ifndef FP8LIN_STAGES2
#define FP8LIN_STAGES2 (FP8LIN_PAIR_BK == 256 ? 3 : 6)
#endif
constexpr int GROUP_M = FP8LIN_GROUP_M;    // 128-row tiles per raster group
constexpr int GROUP_M2 = FP8LIN_GROUP_M2;  // 256-row pair tiles per raster group
constexpr int BAR_BYTES = 256;
constexpr int STAGING_PER_WARP = 32 * 128;            // 32 rows x 128 bytes of output
constexpr int STAGING_BYTES = EPI_WARPS * STAGING_PER_WARP;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + BAR_BYTES + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory per block exceeded");

static_assert(STAGE_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "stage tiles must stay 1024-aligned");
static_assert((2 * STAGES + 2 * ACC + 1) * 8 + 8 <= BAR_BYTES, "barrier area too small");

// Tile t of the raster.  group_m > 0: groups of group_m M blocks, M fastest
// inside a group; group_m = 1 sweeps N fastest (one M band at a time, all of B
// reused), group_m = tiles_m sweeps M fastest over the whole matrix (all of A
// reused).  group_m < 0: groups of -group_m N blocks, N fastest inside a group
// (the group's slice of B reused while A streams through once per group).
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group_m, int& mb, int& nb) {
  if (group_m < 0) {
    const int group_n = -group_m;
    const int group = group_n * tiles_m;
    const int g = t / group;
    const int first_n = g * group_n;
    const int gn = min(group_n, tiles_n - first_n);
    const int r = t - g * group;
    nb = first_n + r % gn;
    mb = r / gn;
    return;
  }
  const int group = group_m * tiles_n;
  const int g = t / group;
  const int first_m = g * group_m;
  const int gm = min(group_m, tiles_m - first_m);
  const int r = t - g * group;
  mb = first_m + r % gm;
  nb = r / gm;
}


// Add one finished TMEM partial (this warp's 32 lanes x EPI_COLS columns
// starting at taddr) into the fp32 register accumulators, round to nearest.
__device__ __forceinline__ void add_partial(float (&acc)[EPI_COLS], uint32_t taddr) {
#pragma unroll
  for (int c = 0; c < EPI_COLS / 8; c += kEpiBatch) {
    uint32_t r[kEpiBatch][8];
#pragma unroll
    for (int b = 0; b < kEpiBatch; ++b) tmem_ld8(taddr + static_cast<uint32_t>((c + b) * 8), r[b]);
    tmem_ld_wait();
#pragma unroll
    for (int b = 0; b < kEpiBatch; ++b)
#pragma unroll
      for (int j = 0; j < 8; j += 2) {  // two round-to-nearest adds per instruction
        float& lo = acc[(c + b) * 8 + j];
        float& hi = acc[(c + b) * 8 + j + 1];
        f2_unpack(f2_add(f2_pack(lo, hi), f2_pack(__uint_as_float(r[b][j]), __uint_as_float(r[b][j + 1]))), lo,
                  hi);
      }
  }
}

// Output kinds of the epilogue.
constexpr int kOutBf16 = 0;
constexpr int kOutF32 = 1;
constexpr int kOutE4M3 = 2;  // FP8 codes of y * s_out (the next stage's scale)
constexpr int kOutE5M2 = 3;

template <int OUT>
__device__ __forceinline__ uint32_t out_cvt_pair(float lo, float hi) {
  return cvt_fp8x2<OUT == kOutE4M3 ? kE4M3 : kE5M2>(lo, hi);
}

// Counters of an FP8 output (the next stage's cast composed into the epilogue).
struct OutQ {
  float qs;      // scale of the output tensor (its delayed scale)
  uint32_t sat;  // |y * qs| > FP8_MAX
  uint32_t und;  // y != 0 and |y * qs| <= half the smallest subnormal
};

// Two values -> two FP8 codes of y * qs (y = acc * factor), folding max|y|
// and the counts of in-range elements.
template <int OUT>
__device__ __forceinline__ uint32_t out_fp8_pair(float a0, float a1, float factor, bool ok0, bool ok1,
                                                 OutQ& q, uint32_t& amax_bits) {
  constexpr float kMax = OUT == kOutE4M3 ? kMaxE4M3 : kMaxE5M2;
  constexpr float kUnd = OUT == kOutE4M3 ? 0.0009765625f : 7.62939453125e-06f;
  const float y0 = __fmul_rn(a0, factor), y1 = __fmul_rn(a1, factor);
  const float p0 = __fmul_rn(y0, q.qs), p1 = __fmul_rn(y1, q.qs);
  if (ok0) {
    amax_bits = max(amax_bits, __float_as_uint(y0) & 0x7FFFFFFFu);
    q.sat += fabsf(p0) > kMax;
    q.und += (y0 != 0.0f) && (fabsf(p0) <= kUnd);
  }
  if (ok1) {
    amax_bits = max(amax_bits, __float_as_uint(y1) & 0x7FFFFFFFu);
    q.sat += fabsf(p1) > kMax;
    q.und += (y1 != 0.0f) && (fabsf(p1) <= kUnd);
  }
  return out_cvt_pair<OUT>(p0, p1);
}

// Eight consecutive values -> eight FP8 codes of y * qs (y = a * factor, both
// products rounded to nearest, two per instruction), folding max|y| and the
// counts of the first `valid` values.  Saturated and underflowed products are
// rare: the eight are first tested together -- the largest |p| against
// FP8_MAX, the smallest against the underflow bound (NaN drops out of both,
// as it fails both per-value tests) -- and counted one by one only when the
// group may hold one.
template <int OUT>
__device__ __forceinline__ uint2 out_fp8_8(const float* a, uint64_t ff, uint64_t qq, int valid, OutQ& q,
                                           uint32_t& amax_bits) {
  constexpr float kMax = OUT == kOutE4M3 ? kMaxE4M3 : kMaxE5M2;
  constexpr float kUnd = OUT == kOutE4M3 ? 0.0009765625f : 7.62939453125e-06f;
  float y[8], p[8];
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const uint64_t yy = f2_mul(f2_pack(a[i], a[i + 1]), ff);
    f2_unpack(yy, y[i], y[i + 1]);
    f2_unpack(f2_mul(yy, qq), p[i], p[i + 1]);
  }
  uint2 w;
  w.x = out_cvt_pair<OUT>(p[0], p[1]) | (out_cvt_pair<OUT>(p[2], p[3]) << 16);
  w.y = out_cvt_pair<OUT>(p[4], p[5]) | (out_cvt_pair<OUT>(p[6], p[7]) << 16);
  if (valid >= 8) {
    float hi = fabsf(p[0]), lo = fabsf(p[0]);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      amax_bits = max(amax_bits, __float_as_uint(y[i]) & 0x7FFFFFFFu);
      hi = fmaxf(hi, fabsf(p[i]));
      lo = fminf(lo, fabsf(p[i]));
    }
    if (hi > kMax) {
#pragma unroll
      for (int i = 0; i < 8; ++i) q.sat += fabsf(p[i]) > kMax;
    }
    if (lo <= kUnd) {
#pragma unroll
      for (int i = 0; i < 8; ++i) q.und += (y[i] != 0.0f) && (fabsf(p[i]) <= kUnd);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < valid) {
        amax_bits = max(amax_bits, __float_as_uint(y[i]) & 0x7FFFFFFFu);
        q.sat += fabsf(p[i]) > kMax;
        q.und += (y[i] != 0.0f) && (fabsf(p[i]) <= kUnd);
      }
    }
  }
  return w;
}

// Dequantise and store one thread's row segment (EPI_COLS columns from colw),
// folding max|stored value| into amax_bits (FP8 outputs: max|y| before the
// output scale, and the counts into q).
template <int OUT>
__device__ __forceinline__ void store_row(const float (&acc)[EPI_COLS], int row, int colw, int M, int N,
                                          void* __restrict__ D, int64_t ldd, float factor, int vec_ok,
                                          uint32_t& amax_bits, OutQ& q) {
  if (row < M) {
#pragma unroll
    for (int c = 0; c < EPI_COLS / 8; ++c) {
      const int col0 = colw + c * 8;
      if (col0 >= N) break;
      const bool full8 = vec_ok && (col0 + 8 <= N);
      if (OUT == kOutF32) {
        float* drow = static_cast<float*>(D) + static_cast<int64_t>(row) * ldd + col0;
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          v[j] = __fmul_rn(acc[c * 8 + j], factor);
          if (col0 + j < N) amax_bits = max(amax_bits, __float_as_uint(v[j]) & 0x7FFFFFFFu);
        }
        if (full8) {
          *reinterpret_cast<float4*>(drow) = make_float4(v[0], v[1], v[2], v[3]);
          *reinterpret_cast<float4*>(drow + 4) = make_float4(v[4], v[5], v[6], v[7]);
        } else {
          for (int j = 0; j < 8; ++j)
            if (col0 + j < N) drow[j] = v[j];
        }
      } else if (OUT == kOutBf16) {
        uint16_t* drow = static_cast<uint16_t*>(D) + static_cast<int64_t>(row) * ldd + col0;
        uint32_t p[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          p[j] = bf16x2_bits(__fmul_rn(acc[c * 8 + 2 * j], factor),
                             __fmul_rn(acc[c * 8 + 2 * j + 1], factor));
        if (full8) {
          const uint32_t m2 = __vmaxu2(__vmaxu2(p[0] & 0x7FFF7FFFu, p[1] & 0x7FFF7FFFu),
                                       __vmaxu2(p[2] & 0x7FFF7FFFu, p[3] & 0x7FFF7FFFu));
          amax_bits = max(amax_bits, max(m2 & 0xFFFFu, m2 >> 16) << 16);
          *reinterpret_cast<uint4*>(drow) = make_uint4(p[0], p[1], p[2], p[3]);
        } else {
          for (int j = 0; j < 8; ++j) {
            if (col0 + j < N) {
              const uint16_t b = static_cast<uint16_t>(p[j >> 1] >> (16 * (j & 1)));
              drow[j] = b;
              amax_bits = max(amax_bits, static_cast<uint32_t>(b & 0x7FFFu) << 16);
            }
          }
        }
      } else {
        uint8_t* drow = static_cast<uint8_t*>(D) + static_cast<int64_t>(row) * ldd + col0;
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t pr = out_fp8_pair<OUT>(acc[c * 8 + 2 * j], acc[c * 8 + 2 * j + 1], factor,
                                                col0 + 2 * j < N, col0 + 2 * j + 1 < N, q, amax_bits);
          w[j >> 1] |= pr << (16 * (j & 1));
        }
        if (full8) {
          *reinterpret_cast<uint2*>(drow) = make_uint2(w[0], w[1]);
        } else {
          for (int j = 0; j < 8; ++j)
            if (col0 + j < N) drow[j] = static_cast<uint8_t>(w[j >> 2] >> (8 * (j & 3)));
        }
      }
    }
  }
}

// Dequantise this warp's 32 rows x EPI_COLS columns (row0 + lane, from colw)
// and write them with TMA stores: each 32-row x 128-byte block (64 bf16, 32
// fp32 or 128 FP8 columns) is staged in the warp's 4 KB buffer in the 128-byte
// swizzled layout (conflict-free 16-byte shared stores), then stored by one
// cp.async.bulk.tensor issued by lane 0.  TMA clips the block at the tensor's
// edges.  With `track` (a tensor records this GEMM's output amax), max|value|
// of in-range elements is folded into amax_bits; FP8 outputs always track
// (max|y| before the output scale, counts into q).
// TMA store of one staged block with an L2 evict-first policy.  No CTA of the
// GEMM reads its output again, so the output lines are the first L2 may give
// up: they leave for DRAM while the GEMM still runs instead of displacing the
// operand tiles that later tiles re-read (1-7 % less DRAM traffic per launch
// on the transformer layer's shapes).
__device__ __forceinline__ void tma_store_2d_evict_first(const CUtensorMap* map, uint32_t src, int32_t c0,
                                                         int32_t c1) {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int OUT>
__device__ __forceinline__ void store_rows_tma(const float (&acc)[EPI_COLS], uint8_t* buf,
                                               const CUtensorMap* tmD, int row0, int colw, int lane,
                                               int M, int N, float factor, uint32_t& amax_bits,
                                               OutQ& q, bool track) {
  constexpr int CPB = OUT == kOutF32 ? 32 : (OUT == kOutBf16 ? 64 : 128);  // columns per block
  constexpr int VPC = CPB / 8;                                               // values per chunk
  const uint32_t sbase = smem_u32(buf);
  const uint64_t ff = f2_pack(factor, factor), qq = f2_pack(q.qs, q.qs);
  const bool row_ok = row0 + lane < M;
#pragma unroll
  for (int b = 0; b < EPI_COLS / CPB; ++b) {
    const int cb = colw + b * CPB;
    if (cb >= N) break;  // warp-uniform
    if (lane == 0) bulk_wait_read_all();  // the previous block has left the buffer
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c0 = cb + j * VPC;
      const float* a = acc + b * CPB + j * VPC;
      uint32_t w[4];
      if (OUT == kOutF32) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          w[t] = __float_as_uint(__fmul_rn(a[t], factor));
          if (track && row_ok && c0 + t < N) amax_bits = max(amax_bits, w[t] & 0x7FFFFFFFu);
        }
      } else if (OUT == kOutBf16) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          float lo = a[2 * t], hi = a[2 * t + 1];
          f2_scale(lo, hi, ff);
          w[t] = bf16x2_bits(lo, hi);
          if (track && row_ok && c0 + 2 * t < N) amax_bits = max(amax_bits, (w[t] & 0x7FFFu) << 16);
          if (track && row_ok && c0 + 2 * t + 1 < N) amax_bits = max(amax_bits, w[t] & 0x7FFF0000u);
        }
      } else {
        const int valid = row_ok ? N - c0 : 0;  // values of this chunk inside the tensor
        const uint2 w01 = out_fp8_8<OUT>(a, ff, qq, valid, q, amax_bits);
        const uint2 w23 = out_fp8_8<OUT>(a + 8, ff, qq, valid - 8, q, amax_bits);
        w[0] = w01.x;
        w[1] = w01.y;
        w[2] = w23.x;
        w[3] = w23.y;
      }
      st_shared_v4(sbase + lane * 128 + ((j ^ (lane & 7)) << 4), w[0], w[1], w[2], w[3]);
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) tma_store_2d_evict_first(tmD, sbase, cb, row0);
  }
}

// ---- activation fused into the epilogue --------------------------------------
// The glue between the two GEMMs of the transformer layer's MLP (FC1 ->
// activation -> FC2), applied to the dequantised fp32 result before it is
// stored, so that FC1 can write FC2's FP8 operand and FC2's dgrad FC1's:
//   kActGelu:  D = out(gelu(y)), and aux (when given) = bf16(gelu'(y)), the
//              derivative the backward multiplies by;
//   kActDgelu: D = out(y * aux), aux = the forward's bf16 gelu'(y).
// The forward computes the derivative from the same exponential as gelu(y),
// so the backward's epilogue does one multiply per value instead of
// re-evaluating the activation.
constexpr int kActNone = 0;
constexpr int kActGelu = 1;
constexpr int kActDgelu = 2;

// GELU in its tanh form, gelu(x) = x/2 * (1 + tanh(u)), u = c (x + a x^3),
// c = sqrt(2/pi), a = 0.044715, through (1 + tanh u)/2 = s = 1 / (1 + e^-2u):
//   gelu(x)  = x * s
//   gelu'(x) = s + 2x * s (1 - s) * c (1 + 3a x^2),   s (1 - s) = e * s^2,
// with e = 2^(-2u log2 e) from the fast exponential (the exponent clamped at
// 80 log2 e, where s < 2^-115) and s from the fast reciprocal.  Two values at a
// time: products and sums as .f32x2 pairs (each half rounded like the scalar
// instruction), the exponential and the reciprocal per value.
constexpr float kGeluC = 0.7978845608028654f;
constexpr float kGeluA = 0.044715f;
constexpr float kGeluA3 = 3.0f * kGeluA;
constexpr float kGeluK = -2.0f * kGeluC * 1.4426950408889634f;  // -2c log2(e)
constexpr float kGeluKMax = 80.0f * 1.4426950408889634f;        // exponent clamp
__device__ __forceinline__ float ex2_approx(float v) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float rcp_approx(float v) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
// (lo, hi) = gelu((lo, hi)); with want_d, (d0, d1) = gelu'((lo, hi)) as well.
template <bool want_d>
__device__ __forceinline__ void gelu_pair(float& lo, float& hi, float& d0, float& d1) {
  const uint64_t xx = f2_pack(lo, hi);
  const uint64_t x2 = f2_mul(xx, xx);
  const uint64_t w = f2_mul(f2_pack(kGeluK, kGeluK), f2_mul(xx, f2_fma(f2_pack(kGeluA, kGeluA), x2,
                                                                        f2_pack(1.0f, 1.0f))));
  float w0, w1;
  f2_unpack(w, w0, w1);
  const uint64_t ee = f2_pack(ex2_approx(fminf(w0, kGeluKMax)), ex2_approx(fminf(w1, kGeluKMax)));
  float p0, p1;
  f2_unpack(f2_add(f2_pack(1.0f, 1.0f), ee), p0, p1);
  const uint64_t ss = f2_pack(rcp_approx(p0), rcp_approx(p1));
  f2_unpack(f2_mul(xx, ss), lo, hi);
  if (want_d) {
    const uint64_t du = f2_mul(f2_pack(2.0f * kGeluC, 2.0f * kGeluC),
                               f2_fma(f2_pack(kGeluA3, kGeluA3), x2, f2_pack(1.0f, 1.0f)));  // 2 u'(x)
    f2_unpack(f2_fma(f2_mul(xx, f2_mul(ee, f2_mul(ss, ss))), du, ss), d0, d1);
  }
}

// Copy this lane's row of the aux block (row0 + lane, 64 bf16 from c0) into
// its 128-byte row of the warp's staging buffer, in the swizzled order the
// output blocks use, with 16-byte cp.async copies through the load/store path
// (the TMA unit is busy streaming the operand stages, and an aux box queued
// behind them waited microseconds).  Out-of-range pieces are zeros (N is a
// multiple of 8, so each 16-byte piece is wholly inside or outside).  Each lane
// copies and later reads only its own row, so no barrier is needed between
// lanes; the caller makes sure the buffer is free.
__device__ __forceinline__ void aux_copy_row(uint32_t sbase, const uint16_t* __restrict__ aux, int64_t ld_aux,
                                             int row0, int c0, int lane, int M, int N) {
  const int row = row0 + lane;
  const uint32_t dst = sbase + lane * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t d = dst + ((j ^ (lane & 7)) << 4);
    const int col = c0 + 8 * j;
    if (row < M && col < N)
      cp_async16(d, aux + static_cast<int64_t>(row) * ld_aux + col);
    else
      st_shared_v4(d, 0u, 0u, 0u, 0u);
  }
  cp_async_commit();
}

// The activation, in place on this warp's accumulated sums (its 32 rows from
// row0, lane = row, EPI_COLS columns from colw), before the values are stored
// (with factor 1 then).  The aux tensor moves through the warp's 4 KB staging
// buffer, 32 rows x 64 bf16 (128 bytes, swizzled like the output blocks) at a
// time: bf16(gelu'(y)) written by TMA stores under kActGelu, gelu' copied in
// per lane under kActDgelu (aux_copy_row).  Under kActDgelu the first block's
// copy was issued at the start of the tile, before the partial sums were
// drained, when colw < N; each lane issues its second block's copy once it has
// used its row of the first.
template <int ACT>
__device__ __forceinline__ void act_prepass(float (&acc)[EPI_COLS], uint8_t* buf, const CUtensorMap* tmAux,
                                            bool has_aux, const uint16_t* __restrict__ aux, int64_t ld_aux,
                                            int row0, int colw, int lane, int M, int N, float factor) {
  const uint32_t sbase = smem_u32(buf);
  const uint64_t ff = f2_pack(factor, factor);
#pragma unroll
  for (int h = 0; h < EPI_COLS / 64; ++h) {
    const int c0 = colw + 64 * h;
    if (c0 >= N) break;  // warp-uniform: nothing from here on is stored
    if (ACT == kActGelu) {
      if (has_aux) {
        if (lane == 0) bulk_wait_read_all();  // earlier stores have left the buffer
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t w[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            float& lo = acc[64 * h + 8 * j + 2 * t];
            float& hi = acc[64 * h + 8 * j + 2 * t + 1];
            float d0, d1;
            f2_scale(lo, hi, ff);
            gelu_pair<true>(lo, hi, d0, d1);
            w[t] = bf16x2_bits(d0, d1);
          }
          st_shared_v4(sbase + lane * 128 + ((j ^ (lane & 7)) << 4), w[0], w[1], w[2], w[3]);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) tma_store_2d(tmAux, sbase, c0, row0);
      } else {
#pragma unroll
        for (int j = 0; j < 64; j += 2) {
          float& lo = acc[64 * h + j];
          float& hi = acc[64 * h + j + 1];
          float d0, d1;
          f2_scale(lo, hi, ff);
          gelu_pair<false>(lo, hi, d0, d1);
        }
      }
    } else {
      // this block's copy was issued earlier: at the start of the tile (h = 0)
      // or once this lane had used its row of the previous block
      cp_async_wait_all();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 v = ld_shared_v4(sbase + lane * 128 + ((j ^ (lane & 7)) << 4));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {  // (y * factor) * gelu'
          float& lo = acc[64 * h + 8 * j + 2 * t];
          float& hi = acc[64 * h + 8 * j + 2 * t + 1];
          f2_unpack(f2_mul(f2_mul(f2_pack(lo, hi), ff), f2_pack(__uint_as_float(w[t] << 16),
                                                                 __uint_as_float(w[t] & 0xFFFF0000u))),
                    lo, hi);
        }
      }
      if (h + 1 < EPI_COLS / 64 && c0 + 64 < N) aux_copy_row(sbase, aux, ld_aux, row0, c0 + 64, lane, M, N);
    }
  }
}

// The output tensor of an FP8-output GEMM: fold the epilogue's counts and
// max|y| (per warp), and record the scale the cast used.
template <int OUT>
__device__ __forceinline__ void out_record(TensorState* s_out, uint32_t amax_bits, const OutQ& q,
                                           int lane, bool writer) {
  const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, amax_bits);
  if (OUT >= kOutE4M3) {
    const uint32_t ws = __reduce_add_sync(0xFFFFFFFFu, q.sat);
    const uint32_t wu = __reduce_add_sync(0xFFFFFFFFu, q.und);
    if (lane == 0) {
      if (ws) atomicAdd(&s_out->n_sat, static_cast<unsigned long long>(ws));
      if (wu) atomicAdd(&s_out->n_und, static_cast<unsigned long long>(wu));
    }
    if (writer) {  // one thread of the grid: the cast's scale, for the GEMM that consumes D
      s_out->cast_scale = q.qs;
      s_out->cast_scale_inv = s_out->scale_inv;
      s_out->dtype = OUT == kOutE4M3 ? kE4M3 : kE5M2;
    }
  }
  if (lane == 0) {
    if (wmax != 0u) atomicMax(&s_out->amax_pending, wmax);
    s_out->recorded = 1;
  }
}

template <int OUT, int ACT>
__global__ void __launch_bounds__(THREADS, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmAux,
                    void* __restrict__ D, int64_t ldd, const void* aux, int64_t ld_aux, int M, int N, int K,
                    int tiles_m, int tiles_n, int group_m, uint32_t idesc, const TensorState* sa,
                    const TensorState* sb, TensorState* s_out, uint32_t* err, int vec_ok, int tma_store,
                    int has_aux, uint32_t extra_tx, int alt_k) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* staging = smem + STAGES * STAGE_BYTES;  // 1024-aligned, 4 KB per epilogue warp
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + STAGING_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + ACC;
  uint64_t* drain = tempty + ACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nk = (K + BK - 1) / BK;
  // operand layouts, from the instruction descriptor's major bits
  const bool a_mn = (idesc >> 15) & 1u;
  const bool b_mn = (idesc >> 16) & 1u;
  const uint32_t a_step = a_mn ? 256u : 2u;
  const uint32_t b_step = b_mn ? 256u : 2u;
  const int num_tiles = tiles_m * tiles_n;
  const int work0 = static_cast<int>(blockIdx.x);
  const int work_stride = static_cast<int>(gridDim.x);
  auto coords = [&](int t, int& mb, int& nb) { tile_coords(t, tiles_m, tiles_n, group_m, mb, nb); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < ACC; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Launched with programmatic dependent launch: the set-up above (barriers,
  // TMEM, tensor-map prefetch) may overlap the previous kernel; every global
  // access comes after this wait.  Then the next kernel may begin launching:
  // its CTAs land only on SMs this grid has left, and wait likewise.
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long issued = 0;
      bool ok = true;
      int it = 0;
      for (int t = work0; ok && t < num_tiles; t += work_stride, ++it) {
        int mb, nb;
        coords(t, mb, nb);
        // Every other tile of this CTA takes its K blocks from the end: the
        // operand slices the previous tile read last are then read first, while
        // they are still in L2 (a panel re-read across waves, such as B of a
        // long-K GEMM, then halves its reuse distance).  The MMAs and the
        // epilogue only see the stage order; each TMEM partial still covers 16
        // consecutive K blocks, so the bound on the sum is unchanged.
        const bool rev = alt_k && (it & 1);
        for (int kq = 0; kq < nk; ++kq) {
          const int kb = rev ? nk - 1 - kq : kq;
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          // extra_tx (0 except under fp8_debug_inject_stall) over-states the first
          // stage's bytes: the MMA warp's wait then runs out
          mbar_expect_tx(&full[stage], STAGE_BYTES + (issued == 0 ? extra_tx : 0u));
          uint8_t* sA = smem + stage * STAGE_BYTES;
          // K-major maps take (k, row) coordinates, MN-major maps (m or n, k)
          if (a_mn)
            tma_load_2d(sA, &tmA, &full[stage], mb * BM, kb * BK);
          else
            tma_load_2d(sA, &tmA, &full[stage], kb * BK, mb * BM);
          if (b_mn) {  // two 128-column chunks
            tma_load_2d(sA + A_BYTES, &tmB, &full[stage], nb * BN, kb * BK);
            tma_load_2d(sA + A_BYTES + B_BYTES / 2, &tmB, &full[stage], nb * BN + BN / 2, kb * BK);
          } else {
            tma_load_2d(sA + A_BYTES, &tmB, &full[stage], kb * BK, nb * BN);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(err, kErrTimeoutGemm);
        // let this CTA's copies in flight land before shared memory is released
        const int pending = issued < STAGES ? (int)issued : STAGES;
        for (int i = 1; i <= pending; ++i) {
          int s = stage - i;
          uint32_t ph = phase;
          if (s < 0) {
            s += STAGES;
            ph ^= 1u;
          }
          const uint32_t addr = smem_u32(&full[s]);
          const uint64_t t0 = gtimer();
          while (!mbar_try_wait(addr, ph) && gtimer() - t0 < kTimeoutNs) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int grp = 0;  // partial-sum groups issued so far (selects the TMEM buffer)
      bool ok = true;
      bool issued_any = false;
      for (int t = work0; ok && t < num_tiles; t += work_stride) {
        uint32_t d_tmem = tmem_base;
        int buf = 0;
        for (int kb = 0; kb < nk; ++kb) {
          const int kg = kb % kGroup;
          if (kg == 0) {  // start a fresh partial in the next buffer
            buf = grp & 1;
            const uint32_t bph = (grp >> 1) & 1;
            if (!mbar_wait(&tempty[buf], bph ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
          }
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES);
          const uint64_t adesc = a_mn ? sdesc_sw128_mn(a_addr, A_BYTES) : sdesc_sw128(a_addr);
          const uint64_t bdesc =
              b_mn ? sdesc_sw128_mn(a_addr + A_BYTES, B_BYTES / 2) : sdesc_sw128(a_addr + A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k) {
            // K = 32 further on: 32 bytes inside the swizzled rows (K-major) or
            // 32 rows of 128 bytes (MN-major), in 16-byte descriptor units
            mma_f8(d_tmem, adesc + a_step * k, bdesc + b_step * k, idesc, (kg | k) ? 1u : 0u);
          }
          issued_any = true;
          mma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if (kg == kGroup - 1 || kb == nk - 1) {
            mma_commit(&tfull[buf]);  // partial complete
            ++grp;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(err, kErrTimeoutGemm);
        if (issued_any) {  // retire MMAs in flight before TMEM is freed
          mma_commit(drain);
          const uint32_t addr = smem_u32(drain);
          const uint64_t t0 = gtimer();
          while (!mbar_try_wait(addr, 0) && gtimer() - t0 < kTimeoutNs) {
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue --
    const int quarter = warp & 3;           // TMEM lanes this warp may read
    const int half = (warp - 2) >> 2;       // which 128 of the 256 columns
    const float factor = __fmul_rn(sa->cast_scale_inv, sb->cast_scale_inv);
    OutQ q{OUT >= kOutE4M3 ? s_out->scale : 1.0f, 0u, 0u};  // the next stage's scale
    const int ngroups = (nk + kGroup - 1) / kGroup;
    uint32_t amax_bits = 0u;
    int grp = 0;
    bool ok = true;
    for (int t = work0; ok && t < num_tiles; t += work_stride) {
      int mb, nb;
      coords(t, mb, nb);
      const int row0 = mb * BM + quarter * 32, colw = nb * BN + half * EPI_COLS;
      if (ACT == kActDgelu && colw < N) {  // the pre-activation lands while the partials are drained
        if (lane == 0) bulk_wait_read_all();  // the last stores have read the buffer
        __syncwarp();
        aux_copy_row(smem_u32(staging + (warp - 2) * STAGING_PER_WARP), static_cast<const uint16_t*>(aux),
                     ld_aux, row0, colw, lane, M, N);
      }
      float acc[EPI_COLS];
#pragma unroll
      for (int j = 0; j < EPI_COLS; ++j) acc[j] = 0.0f;
      for (int g = 0; g < ngroups; ++g, ++grp) {
        const int buf = grp & 1;
        const uint32_t bph = (grp >> 1) & 1;
        int w = 1;
        if (lane == 0) w = mbar_wait_relaxed(&tfull[buf], bph, abort_flag) ? 1 : 0;
        w = __shfl_sync(0xFFFFFFFFu, w, 0);
        if (!w) {
          if (lane == 0) {
            *abort_flag = 1;
            atomicOr(err, kErrTimeoutGemm);
          }
          ok = false;
          break;
        }
        tc_fence_after();
        add_partial(acc, tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(buf * BN + half * EPI_COLS));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
      }
      if (!ok) {
        if (ACT == kActDgelu) cp_async_wait_all();  // the prefetched block lands before the buffer is released
        break;
      }
      float out_factor = factor;
      if (ACT != kActNone) {  // acc becomes the values to store
        act_prepass<ACT>(acc, staging + (warp - 2) * STAGING_PER_WARP, &tmAux, has_aux != 0,
                         static_cast<const uint16_t*>(aux), ld_aux, row0, colw, lane, M, N, factor);
        __syncwarp();  // every lane's copies are done before the buffer stages the output
        out_factor = 1.0f;
      }
      if (tma_store)
        store_rows_tma<OUT>(acc, staging + (warp - 2) * STAGING_PER_WARP, &tmD, row0, colw, lane, M, N,
                            out_factor, amax_bits, q, s_out != nullptr);
      else
        store_row<OUT>(acc, row0 + lane, colw, M, N, D, ldd, out_factor, vec_ok, amax_bits, q);
      __syncwarp();
    }
    if ((tma_store || (ACT == kActGelu && has_aux)) && lane == 0)
      bulk_wait_all();  // stores done before shared memory is released
    __syncwarp();
    if (s_out != nullptr) out_record<OUT>(s_out, amax_bits, q, lane, blockIdx.x == 0 && warp == 2 && lane == 0);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Pair kernel: a cluster of two CTAs (the two SMs of a TPC) computes a 256x256
// output tile with tcgen05.mma.cta_group::2 (M=256, N=256, K=32).  CTA r loads
// A rows [128r, 128r+128) and B rows [128r, 128r+128) of the tile -- half of the
// B bytes a single CTA would need per output -- into a 3-stage ring of 256-byte
// K stages (FP8LIN_PAIR_BK=128: a 6-stage ring of 128-byte stages); both
// halves' TMA loads count on the leader's (rank 0) stage barrier.  The leader
// alone issues the MMAs; each stage's release and each finished partial are
// signalled to both CTAs with a multicast tcgen05.commit; each CTA's eight
// epilogue warps drain its own TMEM (rows 128r..128r+127 of the tile) and tell
// the leader through a remote arrive that the partial buffer is free.
// ---------------------------------------------------------------------------
constexpr int BM2 = 256;                 // pair tile rows (128 per CTA)
// K bytes per stage.  256: eight MMAs per stage wait and commit once, which the
// tensor pipe needs to run near its peak -- with four per stage the fixed cost
// of each stage's wait and commit held the MMA stream to about 3.3 PFLOP/s
// (timing copies of the kernel issuing each stage's MMAs twice ran at 4.4-4.6).
constexpr int BK2 = FP8LIN_PAIR_BK;
static_assert(BK2 == 128 || BK2 == 256, "pair stage: 128 or 256 K bytes");
constexpr int KSUB2 = BK2 / 128;         // 128-byte K boxes of a K-major operand per stage
constexpr int kGroup2 = kGroup * BK / BK2;  // stages per TMEM partial (K = 2048 either way)
static_assert(kGroup2 >= 1 && kGroup2 * BK2 == kGroup * BK, "promotion interval");
constexpr int STAGES2 = FP8LIN_STAGES2;
constexpr int HALF_BYTES = 128 * BK2;    // A or B half per CTA per stage
constexpr int STAGE2_BYTES = 2 * HALF_BYTES;
constexpr int SMEM2_BYTES = STAGES2 * STAGE2_BYTES + STAGING_BYTES + BAR_BYTES + 1024;
static_assert(SMEM2_BYTES <= 232448, "shared memory per block exceeded");
static_assert((2 * STAGES2 + 2 * ACC + 1 + EPI_WARPS) * 8 + 8 <= BAR_BYTES, "barrier area too small");
static_assert(STAGES2 * STAGE2_BYTES >= EPI_WARPS * EPI_COLS * 32 * 4, "split-tail landing zone");

// The two-CTA kernel's work, visited in the same order by every role of a
// cluster.  Whole tiles first: tile t < dp_tiles belongs to cluster t mod
// nclusters (dp_tiles is a multiple of nclusters, so every cluster has the
// same number).  Then the split tail: the last sk_tiles tiles' TMEM partials
// ("groups", G per tile: 2048 of K each) are numbered tile by tile, and
// cluster c takes the contiguous run [c U / nclusters, (c+1) U / nclusters) of
// the U = sk_tiles * G, cut at tile edges into pieces [g0, g1) of one tile.
// A piece with g0 > 0 ("helper", only ever a cluster's first split piece)
// sums its groups and leaves the sum in the cluster's workspace slot; the
// piece with g0 = 0 ("owner") adds its helpers' sums, in cluster order, to its
// own and stores the tile.  So the tail wave's work is shared by every
// cluster instead of leaving the clusters without a last tile idle.
struct PairPieces {
  int t, nclusters, dp_tiles, G, u, u_end;
  __device__ PairPieces(int cluster, int nclusters_, int dp_tiles_, int G_, int sk_units)
      : t(cluster), nclusters(nclusters_), dp_tiles(dp_tiles_), G(G_),
        u(static_cast<int>(static_cast<int64_t>(cluster) * sk_units / nclusters_)),
        u_end(static_cast<int>(static_cast<int64_t>(cluster + 1) * sk_units / nclusters_)) {}
  __device__ bool next(int& tile, int& g0, int& g1, bool& split) {
    if (t < dp_tiles) {
      tile = t;
      g0 = 0;
      g1 = G;
      split = false;
      t += nclusters;
      return true;
    }
    if (u >= u_end) return false;
    tile = dp_tiles + u / G;
    g0 = u % G;
    g1 = min(G, g0 + (u_end - u));
    split = true;
    u += g1 - g0;
    return true;
  }
};

// A CTA leaving a launch that split tiles: the last one out resets the exit
// count and advances the epoch.  (Out of line: inlined at the kernel's end it
// made the allocator spill in the epilogue.)
__device__ __noinline__ void split_epoch_exit(uint32_t* sk_sync) {
  if (atomicAdd(sk_sync + 1, 1u) == gridDim.x - 1) {
    sk_sync[1] = 0u;
    atomicAdd(sk_sync, 1u);
  }
}

template <int OUT, int ACT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    fp8_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmAux,
                         void* __restrict__ D, int64_t ldd, const void* aux, int64_t ld_aux, int M, int N, int K,
                         int tiles_m, int tiles_n, int group_m, uint32_t idesc, const TensorState* sa,
                         const TensorState* sb, TensorState* s_out, uint32_t* err, int vec_ok, int tma_store,
                         int has_aux, uint32_t extra_tx, int alt_k, float* __restrict__ sk_ws,
                         uint32_t* sk_flags, uint32_t* sk_sync, int sk_tiles) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* staging = smem + STAGES2 * STAGE2_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + STAGING_BYTES);
  uint64_t* empty = full + STAGES2;
  uint64_t* tfull = empty + STAGES2;
  uint64_t* tempty = tfull + ACC;
  uint64_t* drain = tempty + ACC;
  uint64_t* fixbar = drain + 1;  // per epilogue warp: its split-tail copy landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fixbar + EPI_WARPS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0 = leader
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;
  const int num_tiles = tiles_m * tiles_n;
  const int nk = (K + BK2 - 1) / BK2;
  const int G = (nk + kGroup2 - 1) / kGroup2;  // TMEM partials per tile
  const int dp_tiles = num_tiles - sk_tiles;   // whole tiles (see PairPieces)
  const int sk_units = sk_tiles * G;
  // The split tail's flags carry the launch epoch plus one.  The epoch lives
  // in device memory (sk_sync[0]) and advances when the last CTA of a launch
  // leaves (sk_sync[1] counts them), so every CTA reads the same value during
  // the launch, a later launch -- or a replay of a captured one -- never
  // matches a flag an earlier one left, and nothing needs resetting after a
  // time-out.  (Read where it is used, to keep it out of the registers.)
  auto sk_seq = [sk_sync]() { return *reinterpret_cast<volatile uint32_t*>(sk_sync) + 1u; };
  // operand layouts, from the instruction descriptor's major bits; either way
  // each CTA holds one 128-element chunk of A (its rows) and of B.  A K-major
  // half is KSUB2 swizzled [128 rows][128 B] boxes side by side in K; an
  // MN-major half is one [BK2 K rows][128 B] box.
  const bool a_mn = (idesc >> 15) & 1u;
  const bool b_mn = (idesc >> 16) & 1u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES2; ++s) {
      mbar_init(&full[s], 1);   // leader: one arrive.expect_tx, both halves' bytes
      mbar_init(&empty[s], 1);  // one multicast commit per use
    }
    for (int a = 0; a < ACC; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * EPI_WARPS);  // leader: epilogue warps of both CTAs
    }
    mbar_init(drain, 1);
    for (int w = 0; w < EPI_WARPS; ++w) mbar_init(&fixbar[w], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc2(tmem_slot, TMEM_COLS);
    tmem_relinquish2();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers exist before anyone signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Launched with programmatic dependent launch: the set-up above (barriers,
  // TMEM, tensor-map prefetch) may overlap the previous kernel; every global
  // access comes after this wait.  Then the next kernel may begin launching:
  // its CTAs land only on SMs this grid has left, and wait likewise.
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long issued = 0;
      bool ok = true;
      PairPieces pieces(cluster, nclusters, dp_tiles, G, sk_units);
      int t, g0, g1;
      bool split;
      for (int it = 0; ok && pieces.next(t, g0, g1, split); ++it) {
        int mb, nb;
        tile_coords(t, tiles_m, tiles_n, group_m, mb, nb);
        // whole tiles alternate their K direction as in the one-CTA kernel's
        // producer; split pieces run ascending
        const bool rev = alt_k && !split && (it & 1);
        const int kq1 = min(nk, g1 * kGroup2);
        for (int kq = g0 * kGroup2; kq < kq1; ++kq) {
          const int kb = rev ? nk - 1 - kq : kq;
          // the stage barriers complete through the async proxy (TMA transaction
          // bytes, tcgen05.commit): a CTA-scope acquire is enough (measured up
          // to 2 % faster than a cluster-scope one)
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t leader_full = mapa_shared(smem_u32(&full[stage]), 0);
          // extra_tx (0 except under fp8_debug_inject_stall) over-states the first
          // stage's bytes: the MMA issuer's wait then runs out
          if (rank == 0) mbar_expect_tx(&full[stage], 2 * STAGE2_BYTES + (issued == 0 ? extra_tx : 0u));
          uint8_t* sA = smem + stage * STAGE2_BYTES;
          const int m0 = mb * BM2 + 128 * (int)rank, n0 = nb * BN + 128 * (int)rank;
          const int k0 = kb * BK2;  // boxes past K read zeros
          if (a_mn)
            tma_load_2d_pair(sA, &tmA, leader_full, m0, k0);
          else
            for (int h = 0; h < KSUB2; ++h)
              tma_load_2d_pair(sA + h * (128 * 128), &tmA, leader_full, k0 + 128 * h, m0);
          if (b_mn)
            tma_load_2d_pair(sA + HALF_BYTES, &tmB, leader_full, n0, k0);
          else
            for (int h = 0; h < KSUB2; ++h)
              tma_load_2d_pair(sA + HALF_BYTES + h * (128 * 128), &tmB, leader_full, k0 + 128 * h, n0);
          ++issued;
          if (++stage == STAGES2) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(err, kErrTimeoutGemm);
      }
      if (!ok && rank == 0) {
        // the leader's stage barriers count both CTAs' copies: let them land
        const int pending = issued < STAGES2 ? (int)issued : STAGES2;
        for (int i = 1; i <= pending; ++i) {
          int s = stage - i;
          uint32_t ph = phase;
          if (s < 0) {
            s += STAGES2;
            ph ^= 1u;
          }
          const uint32_t addr = smem_u32(&full[s]);
          const uint64_t t0 = gtimer();
          while (!mbar_try_wait_cl(addr, ph) && gtimer() - t0 < kTimeoutNs) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------- MMA issuer (leader only) --
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int grp = 0;
      bool ok = true;
      bool issued_any = false;
      PairPieces pieces(cluster, nclusters, dp_tiles, G, sk_units);
      int t, g0, g1;
      bool split;
      while (ok && pieces.next(t, g0, g1, split)) {
        uint32_t d_tmem = tmem_base;
        int buf = 0;
        const int kb1 = min(nk, g1 * kGroup2);
        for (int kb = g0 * kGroup2; kb < kb1; ++kb) {
          const int kg = kb % kGroup2;
          if (kg == 0) {
            buf = grp & 1;
            const uint32_t bph = (grp >> 1) & 1;
            if (!mbar_wait_cl(&tempty[buf], bph ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
          }
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * STAGE2_BYTES);
          const uint32_t b_addr = a_addr + HALF_BYTES;
#pragma unroll
          for (int k = 0; k < BK2 / 32; ++k) {
            // K = 32 further on: 32 bytes inside a K-major box's swizzled rows
            // (the next box every four steps), or 32 K rows of 128 bytes
            const uint64_t ad = a_mn ? sdesc_sw128_mn(a_addr, HALF_BYTES) + 256u * k
                                     : sdesc_sw128(a_addr + (k >> 2) * (128 * 128)) + 2u * (k & 3);
            const uint64_t bd = b_mn ? sdesc_sw128_mn(b_addr, HALF_BYTES) + 256u * k
                                     : sdesc_sw128(b_addr + (k >> 2) * (128 * 128)) + 2u * (k & 3);
            mma_f8_pair(d_tmem, ad, bd, idesc, (kg | k) ? 1u : 0u);
          }
          issued_any = true;
          mma_commit_pair(&empty[stage], 0x3);
          if (++stage == STAGES2) {
            stage = 0;
            phase ^= 1u;
          }
          if (kg == kGroup2 - 1 || kb == kb1 - 1) {
            mma_commit_pair(&tfull[buf], 0x3);
            ++grp;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(err, kErrTimeoutGemm);
        if (issued_any) {
          mma_commit_pair(drain, 0x1);
          const uint32_t addr = smem_u32(drain);
          const uint64_t t0 = gtimer();
          while (!mbar_try_wait_cl(addr, 0) && gtimer() - t0 < kTimeoutNs) {
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue --
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const float factor = __fmul_rn(sa->cast_scale_inv, sb->cast_scale_inv);
    OutQ q{OUT >= kOutE4M3 ? s_out->scale : 1.0f, 0u, 0u};  // the next stage's scale
    const int ew = warp - 2;  // this warp's share of a split tile's workspace slot and flags
    uint32_t fix_phase = 0u;  // parity of this warp's next split-tail copy
    uint32_t amax_bits = 0u;
    int grp = 0;
    bool ok = true;
    PairPieces pieces(cluster, nclusters, dp_tiles, G, sk_units);
    int t, g0, g1;
    bool split;
    while (ok && pieces.next(t, g0, g1, split)) {
      int mb, nb;
      tile_coords(t, tiles_m, tiles_n, group_m, mb, nb);
      const int row0 = mb * BM2 + 128 * (int)rank + quarter * 32, colw = nb * BN + half * EPI_COLS;
      // (the activation variants never split: the launcher keeps their tails
      // whole, and their epilogue needs the registers)
      const bool helper = ACT == kActNone && g0 > 0;                     // leaves its sum for the tile's owner
      const bool owner = ACT == kActNone && split && g0 == 0 && g1 < G;  // adds its helpers' sums, then stores
      if (ACT == kActDgelu && !helper && colw < N) {  // the pre-activation lands while the partials are drained
        if (lane == 0) bulk_wait_read_all();  // the last stores have read the buffer
        __syncwarp();
        aux_copy_row(smem_u32(staging + (warp - 2) * STAGING_PER_WARP), static_cast<const uint16_t*>(aux),
                     ld_aux, row0, colw, lane, M, N);
      }
      float acc[EPI_COLS];
#pragma unroll
      for (int j = 0; j < EPI_COLS; ++j) acc[j] = 0.0f;
      for (int g = g0; g < g1; ++g, ++grp) {
        const int buf = grp & 1;
        const uint32_t bph = (grp >> 1) & 1;
        int w = 1;
        if (lane == 0) w = mbar_wait_cl_relaxed(&tfull[buf], bph, abort_flag) ? 1 : 0;
        w = __shfl_sync(0xFFFFFFFFu, w, 0);
        if (!w) {
          if (lane == 0) {
            *abort_flag = 1;
            atomicOr(err, kErrTimeoutGemm);
          }
          ok = false;
          break;
        }
        tc_fence_after();
        add_partial(acc, tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(buf * BN + half * EPI_COLS));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&tempty[buf]), 0));
      }
      if (!ok) {
        if (ACT == kActDgelu && !helper) cp_async_wait_all();  // the prefetched block lands before the buffer is released
        break;
      }
      if (helper) {
        // this cluster's slot: [rank][epilogue warp][column / 4][lane][4]
        // floats, 512 contiguous bytes per warp store; the flag is published
        // after every lane's stores
        float4* ws = reinterpret_cast<float4*>(
                         sk_ws + (static_cast<size_t>(cluster * 2 + static_cast<int>(rank)) * EPI_WARPS + ew) *
                                     (EPI_COLS * 32)) + lane;
#pragma unroll
        for (int j = 0; j < EPI_COLS / 4; ++j)
          __stcg(ws + j * 32, make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]));
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(sk_flags + (cluster * 2 + static_cast<int>(rank)) * EPI_WARPS + ew, sk_seq());
        continue;
      }
      if (owner) {
        // the helpers of this tile: the next clusters whose shares start inside
        // it, in order (an empty share has no piece)
        // (u0(h) = h U / nclusters < 2^32: U < 76 * 2^19 for K <= 2^30)
        const uint32_t tile_end = static_cast<uint32_t>((t - dp_tiles + 1) * G);
        const uint32_t su = static_cast<uint32_t>(sk_units), nc = static_cast<uint32_t>(nclusters);
        for (int h = cluster + 1; h < nclusters; ++h) {
          const uint32_t hu0 = static_cast<uint32_t>(h) * su / nc;
          if (hu0 >= tile_end) break;
          if ((static_cast<uint32_t>(h) + 1u) * su / nc == hu0) continue;
          const uint32_t* flag = sk_flags + (h * 2 + static_cast<int>(rank)) * EPI_WARPS + ew;
          int w = 1;
          if (lane == 0) w = flag_wait_gpu(flag, sk_seq(), abort_flag) ? 1 : 0;
          w = __shfl_sync(0xFFFFFFFFu, w, 0);
          if (!w) {
            if (lane == 0) {
              *abort_flag = 1;
              atomicOr(err, kErrTimeoutGemm);
            }
            ok = false;
            break;
          }
          // The helper's 16 KB lands by one bulk copy in this warp's part of
          // the stage buffers: the owner piece is the cluster's last, and its
          // last partial's commit means every MMA that read them has completed.
          const uint32_t land = smem_u32(smem) + static_cast<uint32_t>(ew * EPI_COLS * 32 * 4);
          if (lane == 0) {
            fence_async_global();  // the acquired data, before the async-proxy read
            mbar_expect_tx(&fixbar[ew], EPI_COLS * 32 * 4);
            bulk_load(smem + ew * EPI_COLS * 32 * 4,
                      sk_ws + (static_cast<size_t>(h * 2 + static_cast<int>(rank)) * EPI_WARPS + ew) * (EPI_COLS * 32),
                      EPI_COLS * 32 * 4, &fixbar[ew]);
          }
          w = mbar_wait(&fixbar[ew], fix_phase, abort_flag) ? 1 : 0;
          w = __all_sync(0xFFFFFFFFu, w);
          if (!w) {
            if (lane == 0) {
              *abort_flag = 1;
              atomicOr(err, kErrTimeoutGemm);
              // the copy lands (bounded) before the CTA may leave
              const uint32_t addr = smem_u32(&fixbar[ew]);
              const uint64_t t0 = gtimer();
              while (!mbar_try_wait(addr, fix_phase) && gtimer() - t0 < kTimeoutNs) {
              }
            }
            ok = false;
            break;
          }
          fix_phase ^= 1u;
#pragma unroll
          for (int j = 0; j < EPI_COLS / 4; ++j) {
            const uint4 v = ld_shared_v4(land + static_cast<uint32_t>((j * 32 + lane) * 16));
            acc[4 * j] = __fadd_rn(acc[4 * j], __uint_as_float(v.x));
            acc[4 * j + 1] = __fadd_rn(acc[4 * j + 1], __uint_as_float(v.y));
            acc[4 * j + 2] = __fadd_rn(acc[4 * j + 2], __uint_as_float(v.z));
            acc[4 * j + 3] = __fadd_rn(acc[4 * j + 3], __uint_as_float(v.w));
          }
          __syncwarp();  // every lane has read the landing zone before the next copy
        }
        if (!ok) {
          if (ACT == kActDgelu) cp_async_wait_all();
          break;
        }
      }
      float out_factor = factor;
      if (ACT != kActNone) {  // acc becomes the values to store
        act_prepass<ACT>(acc, staging + (warp - 2) * STAGING_PER_WARP, &tmAux, has_aux != 0,
                         static_cast<const uint16_t*>(aux), ld_aux, row0, colw, lane, M, N, factor);
        __syncwarp();  // every lane's copies are done before the buffer stages the output
        out_factor = 1.0f;
      }
      if (tma_store)
        store_rows_tma<OUT>(acc, staging + (warp - 2) * STAGING_PER_WARP, &tmD, row0, colw, lane, M, N,
                            out_factor, amax_bits, q, s_out != nullptr);
      else
        store_row<OUT>(acc, row0 + lane, colw, M, N, D, ldd, out_factor, vec_ok, amax_bits, q);
      __syncwarp();
    }
    if ((tma_store || (ACT == kActGelu && has_aux)) && lane == 0)
      bulk_wait_all();  // stores done before shared memory is released
    __syncwarp();
    if (s_out != nullptr) out_record<OUT>(s_out, amax_bits, q, lane, blockIdx.x == 0 && warp == 2 && lane == 0);
  }

  tc_fence_before();
  cluster_sync_all();  // no signal may target a CTA that has left
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc2(tmem_base, TMEM_COLS);
  }
  // the last CTA out advances the epoch: every CTA has read it by then (only
  // launches that split a tile use the flags, so only they need to)
  if (sk_tiles > 0 && sk_sync != nullptr && threadIdx.x == 0) split_epoch_exit(sk_sync);
}


// Split tail of the two-CTA kernel (PairPieces); FP8LIN_GEMM_SPLIT_TAIL=0
// turns it off (for comparison).
bool split_tail_enabled() {
  static const bool v = [] {
    const char* e = getenv("FP8LIN_GEMM_SPLIT_TAIL");
    return !(e != nullptr && strcmp(e, "0") == 0);
  }();
  return v;
}

// Kernel choice, read once from the environment (FP8LIN_GEMM_KERNEL):
//   unset   the two-CTA kernel (cta_group::2, 256x256 tiles) for M > 128, and
//           for M <= 128 when few tiles meet a long K (see launch_t);
//   "one"   the one-CTA kernel for every shape.
// Otherwise M <= 128 runs the one-CTA kernel.
enum class KernelChoice { kOne, kPair };
KernelChoice kernel_choice() {
  static const KernelChoice k = [] {
    const char* v = getenv("FP8LIN_GEMM_KERNEL");
    if (v != nullptr && strcmp(v, "one") == 0) return KernelChoice::kOne;
    return KernelChoice::kPair;
  }();
  return k;
}

// Per-device launch set-up of one output kind and activation: the kernels' shared-memory
// opt-in, and how many two-CTA clusters can be resident at once (a persistent
// grid must fit at once; SMs pair up inside a GPC, so this can be fewer than
// num_sms / 2).  Taken on a device's first launch.
template <int OUT, int ACT>
cudaError_t device_setup(cudaStream_t s, int* pair_resident) {
  static PerDevice setup;
  return setup.run(
      [&](int& resident) {
        cudaError_t e =
            cudaFuncSetAttribute(fp8_gemm_kernel<OUT, ACT>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e == cudaSuccess)
          e = cudaFuncSetAttribute(fp8_gemm_pair_kernel<OUT, ACT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   SMEM2_BYTES);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t c = {};
        c.blockDim = dim3(THREADS);
        c.gridDim = dim3(2);
        c.dynamicSmemBytes = SMEM2_BYTES;
        c.stream = s;
        if (cudaOccupancyMaxActiveClusters(&resident, fp8_gemm_pair_kernel<OUT, ACT>, &c) != cudaSuccess)
          resident = 0;
        cudaGetLastError();
        return cudaSuccess;
      },
      pair_resident);
}

// L2 capacity of the current device (queried once per device).
int l2_cache_bytes() {
  static PerDevice l2;
  int bytes = 0;
  if (l2.run(
          [](int& v) {
            int dev = 0;
            cudaGetDevice(&dev);
            if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess) v = 0;
            cudaGetLastError();
            return cudaSuccess;
          },
          &bytes) != cudaSuccess)
    return 0;
  return bytes;
}

// Raster group of a GEMM (tile_coords' group_m): keep one operand's panel, or
// each part of it in turn, resident in L2 while the other streams through.
// A panel of up to 30 % of the L2 stays across waves; 50-67 MB panels (B of
// the N = 4096, K >= 12288 shapes) did not: read once per N-fastest sweep they
// were re-read every wave (2.5x the algorithmic DRAM bytes on 8192 x 4096 x
// 16384).  So:
//  * B's panel (N x K bytes) no larger than A's and within 60 % of the L2: B is
//    split into the fewest equal column groups of at most 30 % each, taken one
//    after another with N fastest inside a group; A streams through once per
//    group (one group: every A band read once, all of B resident);
//  * else A's panel within 60 %: the same with M groups (one group: M fastest
//    over all of M);
//  * else the default grouping.
// The order changes no result: every tile is computed alike.
// FP8LIN_GEMM_RASTER=group keeps the default grouping for every shape, and
// FP8LIN_GEMM_RASTER=n<k> groups k N blocks (for comparison).
int raster_group(const GemmArgs& g, int tiles_m, int tiles_n, int l2_bytes, int fallback) {
  static const int forced = [] {
    const char* v = getenv("FP8LIN_GEMM_RASTER");
    if (v == nullptr) return 0;
    if (strcmp(v, "group") == 0) return 1;
    if (v[0] == 'n' && atoi(v + 1) > 0) return -atoi(v + 1);
    return 0;
  }();
  if (forced == 1) return fallback;
  if (forced < 0) return forced;
  const double resident = 0.3 * l2_bytes;
  const double a_bytes = static_cast<double>(g.M) * g.K, b_bytes = static_cast<double>(g.N) * g.K;
  if (resident <= 0.0) return fallback;
  if (b_bytes <= a_bytes && b_bytes <= 2.0 * resident) {
    const int parts = static_cast<int>(std::ceil(b_bytes / resident));
    return parts <= 1 ? 1 : -((tiles_n + parts - 1) / parts);
  }
  if (a_bytes <= 2.0 * resident) {
    const int parts = std::max(1, static_cast<int>(std::ceil(a_bytes / resident)));
    return (tiles_m + parts - 1) / parts;
  }
  return fallback;
}

template <int OUT, int ACT>
cudaError_t launch_t(const GemmArgs& g, int num_sms, cudaStream_t s, const char** detail) {
  const int l2_bytes = l2_cache_bytes();
  const bool pair_allowed = num_sms >= 2 && kernel_choice() == KernelChoice::kPair;
  bool pair = pair_allowed && g.M > BM;
  if (!pair && pair_allowed && ACT == kActNone && split_tail_enabled() && g.sk_ws != nullptr) {
    // M <= 128 fills a 256-row pair tile only half; but when the one-CTA grid
    // would leave three quarters of the SMs idle on a long K (4 or more
    // 2048-deep partials per tile), the pair kernel's split tail (every pair
    // sharing the tiles' partials) finishes sooner.
    const int64_t tiles_one = ((g.M + BM - 1) / BM) * ((g.N + BN - 1) / BN);
    const int64_t groups = ((g.K + BK2 - 1) / BK2 + kGroup2 - 1) / kGroup2;
    pair = 4 * tiles_one <= num_sms && groups >= 4;
  }
  int resident = 0;
  const cudaError_t setup_err = device_setup<OUT, ACT>(s, &resident);
  if (setup_err != cudaSuccess) return setup_err;
  CUtensorMap ma, mb;
  // K-major: boxes of 128 K bytes x rows; pair: both operands are loaded as
  // 128-row halves.  MN-major: boxes of 128 M or N bytes x 128 (pair: 256) K
  // rows (B as two such chunks, or one per CTA under pair).
  const int mn_box_k = pair ? BK2 : BK;  // K rows of an MN-major box
  const bool maps_ok =
      (g.a_mn ? make_map(&ma, g.A, g.M, g.K, g.lda, 128, mn_box_k) : make_map(&ma, g.A, g.K, g.M, g.lda, BK, BM)) &&
      (g.b_mn ? make_map(&mb, g.B, g.N, g.K, g.ldb, 128, mn_box_k)
              : make_map(&mb, g.B, g.K, g.N, g.ldb, BK, pair ? 128 : BN));
  if (!maps_ok) {
    if (detail) *detail = "cuTensorMapEncodeTiled failed (driver entry point or arguments)";
    return cudaErrorInvalidValue;
  }
  const int bm = pair ? BM2 : BM;
  const int tiles_m = static_cast<int>((g.M + bm - 1) / bm);
  const int tiles_n = static_cast<int>((g.N + BN - 1) / BN);
  const int tiles = tiles_m * tiles_n;
  const int group_m = raster_group(g, tiles_m, tiles_n, l2_bytes, pair ? GROUP_M2 : GROUP_M);
  // instruction descriptor: fp32 accumulate, A/B formats, A/B major (bit 15,
  // 16: 1 = MN-major), N >> 3 at bit 17, M >> 4 at bit 24
  const uint32_t idesc = (1u << 4) | (static_cast<uint32_t>(g.a_dtype) << 7) |
                         (static_cast<uint32_t>(g.b_dtype) << 10) | (g.a_mn ? 1u << 15 : 0u) |
                         (g.b_mn ? 1u << 16 : 0u) |
                         (static_cast<uint32_t>(BN >> 3) << 17) |
                         (static_cast<uint32_t>(bm >> 4) << 24);
  const int esize = OUT == kOutF32 ? 4 : (OUT == kOutBf16 ? 2 : 1);
  const int vec_ok = ((g.ldd * esize) % 16 == 0) && ((reinterpret_cast<uintptr_t>(g.D) & 15) == 0);
  CUtensorMap md;
  memset(&md, 0, sizeof md);
  const int tma_store = make_out_map(&md, g.D, g.M, g.N, g.ldd, esize) ? 1 : 0;
  // the activation's aux tensor (bf16 [M, N]): GELU stores it from the epilogue
  // warps' staging buffers in 32-row x 64-column boxes; GELU' copies it in per
  // lane (no map needed)
  CUtensorMap maux;
  memset(&maux, 0, sizeof maux);
  const int has_aux = ACT != kActNone && g.aux != nullptr ? 1 : 0;
  if (has_aux && ACT == kActGelu && !make_out_map(&maux, g.aux, g.M, g.N, g.ld_aux, 2)) {
    if (detail) *detail = "cuTensorMapEncodeTiled failed for the activation's aux tensor";
    return cudaErrorInvalidValue;
  }
  const int M = static_cast<int>(g.M), N = static_cast<int>(g.N), K = static_cast<int>(g.K);
  // K direction alternating per tile (the producers); FP8LIN_GEMM_KDIR=fwd
  // keeps every tile in ascending K (for comparison)
  static const int alt_k = [] {
    const char* v = getenv("FP8LIN_GEMM_KDIR");
    return v != nullptr && strcmp(v, "fwd") == 0 ? 0 : 1;
  }();
  if (pair) {
    const int cap = resident > 0 && resident < num_sms / 2 ? resident : num_sms / 2;
    int clusters = tiles < cap ? tiles : cap;
    // Split tail (PairPieces): the last, partial wave of tiles -- all of them
    // when there are fewer tiles than clusters -- is shared out by TMEM partial
    // across every resident cluster, when that shortens it and the wave would
    // leave at least half of the clusters idle.  (With fewer idle clusters the
    // busy ones run faster on the power and bandwidth the idle ones leave:
    // at 8192 x 4096 x 16384, 56 busy clusters of 76 took 4.3 us per 2048 of
    // K against 5.5 in full waves, and splitting that tail gained nothing.)
    int sk_tiles = 0;
    const int groups = static_cast<int>(((K + BK2 - 1) / BK2 + kGroup2 - 1) / kGroup2);
    if (ACT == kActNone && split_tail_enabled() && g.sk_ws != nullptr && g.sk_flags != nullptr &&
        cap <= g.sk_slots && groups >= 2) {
      const int rem = tiles % cap;
      if (rem != 0 && 2 * rem <= cap + (tiles < cap ? tiles : 0) && (rem * groups + cap - 1) / cap < groups) {
        sk_tiles = rem;
        clusters = cap;
      }
    }
    return launch_pdl(fp8_gemm_pair_kernel<OUT, ACT>, dim3(2 * clusters), dim3(THREADS), SMEM2_BYTES, s, ma, mb, md,
                      maux, g.D, g.ldd, g.aux, g.ld_aux, M, N, K, tiles_m, tiles_n, group_m, idesc, g.sa, g.sb,
                      g.s_out, g.error, vec_ok, tma_store, has_aux, g.extra_tx, alt_k, g.sk_ws, g.sk_flags,
                      g.sk_flags != nullptr ? g.sk_flags + kSplitSlotFlags * g.sk_slots : nullptr, sk_tiles);
  }
  const int grid = tiles < num_sms ? tiles : num_sms;
  return launch_pdl(fp8_gemm_kernel<OUT, ACT>, dim3(grid), dim3(THREADS), SMEM_BYTES, s, ma, mb, md, maux, g.D,
                    g.ldd, g.aux, g.ld_aux, M, N, K, tiles_m, tiles_n, group_m, idesc, g.sa, g.sb, g.s_out, g.error,
                    vec_ok, tma_store, has_aux, g.extra_tx, alt_k);
}

}  // namespace

void* tma_encoder() {
  static void* fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = p;
  });
  return fn;
}

namespace {
template <int ACT>
cudaError_t launch_act(const GemmArgs& g, int num_sms, cudaStream_t s, const char** detail) {
  switch (g.d_kind) {
    case kOutF32: return launch_t<kOutF32, ACT>(g, num_sms, s, detail);
    case kOutE4M3: return launch_t<kOutE4M3, ACT>(g, num_sms, s, detail);
    case kOutE5M2: return launch_t<kOutE5M2, ACT>(g, num_sms, s, detail);
    default: return launch_t<kOutBf16, ACT>(g, num_sms, s, detail);
  }
}
}  // namespace

cudaError_t launch_gemm(const GemmArgs& g, int num_sms, cudaStream_t s, const char** detail) {
  switch (g.act) {
    case kActGelu: return launch_act<kActGelu>(g, num_sms, s, detail);
    case kActDgelu: return launch_act<kActDgelu>(g, num_sms, s, detail);
    default: return launch_act<kActNone>(g, num_sms, s, detail);
  }
}

}  // namespace fp8lin
