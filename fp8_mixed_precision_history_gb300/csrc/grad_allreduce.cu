// grad_allreduce.cu -- the device steps of an FP8 (E5M2) gradient all-reduce
// with automatic scaling.
//
// "FP8 and low-precision formats" (aiunderstanding.org), use cases: E5M2 for
// gradient communication in distributed training, to cut inter-node
// bandwidth.  "[📪정보] 그저께 나온 논문 대박이네" (mir.rootios.com, a thread on the
// FP8-LM paper): automatic scaling adjusts the tensor scaling factor so that
// gradients stay inside FP8's range during the all-reduce.  Reading taken:
//   1. amax = max over all ranks of max|g| (each rank: grad_amax_kernel, then
//      a MAX all-reduce of one float between the ranks);
//   2. one scale s = 57344 / fp32(world * amax) for every rank, so that the
//      world-way sum of scaled values cannot leave E5M2's range (s = 1 for a
//      zero or non-finite amax; world * amax and s clamp at FLT_MAX);
//   3. each rank casts fp32(g * s) to E5M2 (grad_quantize_kernel);
//   4. reduce-scatter: rank r receives chunk r of every rank's codes and sums
//      them EXACTLY -- every E5M2 value is an integer multiple of 2^-16 below
//      2^32 of them -- then rounds the sum to E5M2 once (nearest, ties to
//      even, saturating; an Inf or NaN code makes the NaN code 0x7E):
//      grad_reduce_f32_kernel up to 128 ranks (two exact fp32 sums, rounded
//      through rounding to odd), grad_reduce_kernel above (integer sums);
//   5. all-gather of the reduced codes;
//   6. result = bf16(fp32(decode(code) * f)), f = 1/s, or fp32((1/s) / world)
//      for the mean (grad_dequantize_kernel).
// One byte per element travels in each of steps 4 and 5, against two per
// element per phase for a bf16 all-reduce.
// No kernel here waits on anything: none can time out.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cfloat>
#include <cstdint>

#include "state.cuh"
#include "tc_ptx.cuh"

namespace fp8lin {
namespace {

constexpr int kThreads = 256;  // the reduce kernel builds its 256-entry table with one thread per entry

__device__ __forceinline__ float shared_scale(const float* amax, int world) {
  const float a = *amax;
  if (!(a > 0.0f) || isinf(a)) return 1.0f;
  float d = __fmul_rn(static_cast<float>(world), a);
  if (isinf(d)) d = FLT_MAX;
  float s = __fdiv_rn(57344.0f, d);
  if (isinf(s)) s = FLT_MAX;
  return s;
}

// The amax and quantise kernels cover the vector once: each thread loads
// kGradU 16-byte vectors (8 bf16 each) before using any of them, so enough
// loads are in flight to keep HBM busy.
constexpr int kGradU = 8;
constexpr int kGradBlockVecs = kThreads * kGradU;  // 16-byte vectors per block

int one_pass_grid(int64_t vecs) {
  return static_cast<int>(std::max<int64_t>(1, (vecs + kGradBlockVecs - 1) / kGradBlockVecs));
}

// ---- 1. amax of a bf16 vector (bit patterns; NaN above Inf) -----------------
__global__ void __launch_bounds__(kThreads) grad_amax_kernel(const uint16_t* __restrict__ g, int64_t n,
                                                             uint32_t* amax_bits) {
  const int64_t nv = n / 8;
  const uint4* g8 = reinterpret_cast<const uint4*>(g);
  const int64_t base = blockIdx.x * static_cast<int64_t>(kGradBlockVecs) + threadIdx.x;
  uint4 v[kGradU];
#pragma unroll
  for (int u = 0; u < kGradU; ++u) {
    const int64_t i = base + u * kThreads;
    v[u] = i < nv ? __ldcs(g8 + i) : make_uint4(0u, 0u, 0u, 0u);
  }
  uint32_t m2 = 0u;
#pragma unroll
  for (int u = 0; u < kGradU; ++u)
    m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(v[u].x & 0x7FFF7FFFu, v[u].y & 0x7FFF7FFFu),
                               __vmaxu2(v[u].z & 0x7FFF7FFFu, v[u].w & 0x7FFF7FFFu)));
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
  if (blockIdx.x == gridDim.x - 1)  // the last n % 8 elements
    for (int64_t i = 8 * nv + threadIdx.x; i < n; i += kThreads) m = max(m, static_cast<uint32_t>(g[i] & 0x7FFFu));
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  __shared__ uint32_t wmax[kThreads / 32];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t b = threadIdx.x < kThreads / 32 ? wmax[threadIdx.x] : 0u;
    b = __reduce_max_sync(0xFFFFFFFFu, b);
    if (threadIdx.x == 0 && b != 0u) atomicMax(amax_bits, b << 16);  // fp32 bits of the bf16 value
  }
}

// ---- 3. E5M2 codes of g * s, zero padding up to padded_n ---------------------
// The grid covers the padded_n / 8 whole eight-code groups; the last block
// also writes the padded_n % 8 codes after them.
__global__ void __launch_bounds__(kThreads) grad_quantize_kernel(const uint16_t* __restrict__ g, int64_t n,
                                                                 const float* amax, int world,
                                                                 uint8_t* __restrict__ codes, int64_t padded_n,
                                                                 float* scale_out) {
  const float s = shared_scale(amax, world);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    scale_out[0] = s;
    scale_out[1] = __fdiv_rn(1.0f, s);
  }
  const int64_t nv = n / 8, pv = padded_n / 8;
  const uint4* g8 = reinterpret_cast<const uint4*>(g);
  uint2* c8 = reinterpret_cast<uint2*>(codes);
  const int64_t base = blockIdx.x * static_cast<int64_t>(kGradBlockVecs) + threadIdx.x;
  uint4 v[kGradU];
#pragma unroll
  for (int u = 0; u < kGradU; ++u) {
    const int64_t i = base + u * kThreads;
    v[u] = i < nv ? __ldcs(g8 + i) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int u = 0; u < kGradU; ++u) {
    const int64_t i = base + u * kThreads;
    if (i < nv) {
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      uint32_t p[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        p[j] = cvt_fp8x2<kE5M2>(__fmul_rn(__uint_as_float(w[j] << 16), s),
                                __fmul_rn(__uint_as_float(w[j] & 0xFFFF0000u), s));
      c8[i] = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
    } else if (i < pv) {  // the ragged end and the zero padding
      uint32_t p[2] = {0u, 0u};
      for (int k = 0; k < 8; ++k) {
        const int64_t e = 8 * i + k;
        if (e < n)
          p[k >> 2] |= (cvt_fp8x2<kE5M2>(__fmul_rn(__uint_as_float(static_cast<uint32_t>(g[e]) << 16), s), 0.0f) &
                        0xFFu)
                       << (8 * (k & 3));
      }
      c8[i] = make_uint2(p[0], p[1]);
    }
  }
  if (blockIdx.x == gridDim.x - 1) {
    const int64_t e = 8 * pv + threadIdx.x;
    if (e < padded_n)
      codes[e] = e < n ? static_cast<uint8_t>(
                             cvt_fp8x2<kE5M2>(__fmul_rn(__uint_as_float(static_cast<uint32_t>(g[e]) << 16), s), 0.0f))
                       : 0;
  }
}

// ---- 4. exact sum of world code vectors, rounded to E5M2 --------------------
// E5M2 code -> value in units of 2^-16: subnormal f (e = 0), else (4 + f) << (e - 1);
// at most 7 * 2^29, so it fits 32 bits.
__device__ __forceinline__ uint32_t e5m2_magnitude_units(uint32_t c) {
  const uint32_t e = (c >> 2) & 31u, f = c & 3u;
  return e == 0u ? f : (4u + f) << (e - 1u);
}
// Round an exact sum (units of 2^-16) to E5M2, nearest with ties to the even
// code, saturating at 57344 (code 0x7B); neg_zero: the sum is -0.
__device__ __forceinline__ uint32_t e5m2_round(int64_t sum, bool neg_zero) {
  if (sum == 0) return neg_zero ? 0x80u : 0x00u;
  const uint32_t sign = sum < 0 ? 0x80u : 0x00u;
  uint64_t m = static_cast<uint64_t>(sum < 0 ? -sum : sum);
  if (m < 8u) return sign | (m < 4u ? static_cast<uint32_t>(m) : (1u << 2) | static_cast<uint32_t>(m - 4u));
  int shift = 63 - __clzll(static_cast<long long>(m)) - 2;  // keep three significant bits
  uint64_t q = m >> shift;
  const uint64_t rem = m & ((uint64_t{1} << shift) - 1u);
  const uint64_t half = uint64_t{1} << (shift - 1);
  if (rem > half || (rem == half && (q & 1u))) ++q;
  if (q == 8u) {
    q = 4u;
    ++shift;
  }
  const uint32_t e = static_cast<uint32_t>(shift) + 1u;
  if (e > 30u) return sign | 0x7Bu;
  return sign | (e << 2) | static_cast<uint32_t>(q - 4u);
}

// Each thread sums 4 consecutive codes (one 32-bit word) of every rank.  A
// code's value is looked up as two signed halves, (units >> 16) and
// (units & 0xFFFF), so that the per-element sums stay exact in 32-bit integers
// for up to 2^15 ranks (FP8_GRAD_MAX_WORLD; each half adds at most 65535 per
// rank); they are joined into one int64 before the rounding.  Negative zeros
// and Inf/NaN codes are tracked four bytes at a time.
__global__ void __launch_bounds__(kThreads) grad_reduce_kernel(const uint8_t* __restrict__ recv, int world,
                                                               int64_t chunk, uint8_t* __restrict__ out) {
  static_assert(kThreads == 256, "one table entry per thread");
  __shared__ int2 tab[256];
  {
    const uint32_t c = threadIdx.x;
    const uint32_t m = e5m2_magnitude_units(c);
    const int hi = static_cast<int>(m >> 16), lo = static_cast<int>(m & 0xFFFFu);
    tab[c] = (c & 0x80u) ? make_int2(-hi, -lo) : make_int2(hi, lo);
  }
  __syncthreads();
  const int64_t n4 = chunk / 4;  // chunk % 16 == 0
  const uint32_t* rw = reinterpret_cast<const uint32_t*>(recv);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    int hi0 = 0, hi1 = 0, hi2 = 0, hi3 = 0, lo0 = 0, lo1 = 0, lo2 = 0, lo3 = 0;
    uint32_t negz = 0xFFFFFFFFu, nan = 0u;  // byte masks
#pragma unroll 4
    for (int r = 0; r < world; ++r) {
      const uint32_t w = __ldcs(rw + static_cast<int64_t>(r) * (chunk / 4) + i);
      negz &= __vcmpeq4(w, 0x80808080u);
      nan |= __vcmpeq4(w & 0x7C7C7C7Cu, 0x7C7C7C7Cu);
      const int2 t0 = tab[w & 0xFFu], t1 = tab[(w >> 8) & 0xFFu], t2 = tab[(w >> 16) & 0xFFu], t3 = tab[w >> 24];
      hi0 += t0.x;
      lo0 += t0.y;
      hi1 += t1.x;
      lo1 += t1.y;
      hi2 += t2.x;
      lo2 += t2.y;
      hi3 += t3.x;
      lo3 += t3.y;
    }
    const int hi[4] = {hi0, hi1, hi2, hi3}, lo[4] = {lo0, lo1, lo2, lo3};
    uint32_t o = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t byte = 8u * j;
      const int64_t sum = (static_cast<int64_t>(hi[j]) << 16) + lo[j];
      const uint32_t c = ((nan >> byte) & 1u) ? 0x7Eu : e5m2_round(sum, (negz >> byte) & 1u);
      o |= c << byte;
    }
    reinterpret_cast<uint32_t*>(out)[i] = o;
  }
}

// The same sum for up to 128 ranks in fp32, also exact: a decoded code v
// (|v| <= 57344, a multiple of 2^-16) is split into its nearest integer
// h = (v + 1.5 * 2^23) - 1.5 * 2^23 and the rest l = v - h (|l| <= 1/2, a
// multiple of 2^-16); both splits are exact.  Over <= 128 ranks the sum of
// the h stays an integer below 2^24 and the sum of the l a multiple of 2^-16
// below 2^6 in magnitude -- both exact in fp32.  Runs on the FP32 pipe with
// no table.
constexpr int kReduceF32MaxWorld = 128;


__device__ __forceinline__ void e5m2x4_values(uint32_t w, float2& f01, float2& f23) {
  // an E5M2 code is the top byte of the binary16 value it encodes
  const uint32_t h01 = __byte_perm(w, 0u, 0x1404), h23 = __byte_perm(w, 0u, 0x3424);
  f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
  f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
}

// E5M2 codes (low byte: the first element) of the exact sums H + L of an
// element pair, packed as .f32x2, by rounding to odd: the sum rounded toward
// zero, with its last bit set where the sum is inexact, is the odd one of the
// two fp32 values around it (or the sum itself).  TwoSum's error term of the
// nearest-rounded sum tells whether it is exact.  A sum rounded to odd with
// at least two more bits than the target rounds to nearest correctly (Boldo
// and Melquiond, "Emulation of FMA and correctly rounded sums: proved
// algorithms using rounding to odd", IEEE TC 2008); fp32 has 24 bits against
// E5M2's 3, at every E5M2 exponent.  A zero sum of -0 addends only (H = +0,
// L = -0) gives -0.  A NaN sum gives the conversion's NaN code.
__device__ __forceinline__ uint64_t f2_add_rz(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint32_t e5m2x2_of_exact_sums(uint64_t H, uint64_t L, uint64_t minus1) {
  const uint64_t s = f2_add(H, L);
  const uint64_t bb = f2_fma(H, minus1, s);                                     // s - H
  const uint64_t e = f2_add(f2_fma(f2_fma(bb, minus1, s), minus1, H),          // H - (s - bb)
                            f2_fma(bb, minus1, L));                             // + (L - bb)
  const uint64_t z = f2_add_rz(H, L);
  float z0, z1, e0, e1, h0, h1, l0, l1;
  f2_unpack(z, z0, z1);
  f2_unpack(e, e0, e1);
  f2_unpack(H, h0, h1);
  f2_unpack(L, l0, l1);
  // negative zero: H = +0 and L = -0
  const uint32_t nz0 = (__float_as_uint(h0) | (__float_as_uint(l0) ^ 0x80000000u)) == 0u ? 0x80000000u : 0u;
  const uint32_t nz1 = (__float_as_uint(h1) | (__float_as_uint(l1) ^ 0x80000000u)) == 0u ? 0x80000000u : 0u;
  const uint32_t r0 = __float_as_uint(z0) | (e0 != 0.0f ? 1u : 0u) | nz0;
  const uint32_t r1 = __float_as_uint(z1) | (e1 != 0.0f ? 1u : 0u) | nz1;
  return cvt_fp8x2<kE5M2>(__uint_as_float(r0), __uint_as_float(r1));
}

constexpr int kReduceBatch = 8;      // ranks whose words are loaded together
constexpr int kReduceCtasPerSm = 5;  // what its registers allow

// Eight codes per thread (one 8-byte word per rank); pairs of elements share
// one packed fp32 instruction (.f32x2), which rounds each half exactly like the
// scalar one.
__global__ void __launch_bounds__(kThreads, kReduceCtasPerSm) grad_reduce_f32_kernel(const uint8_t* __restrict__ recv, int world,
                                                                   int64_t chunk, uint8_t* __restrict__ out) {
  constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
  const uint64_t up = f2_pack(kRound, kRound), down = f2_pack(-kRound, -kRound), minus1 = f2_pack(-1.0f, -1.0f);
  const int64_t n8 = chunk / 8;
  const uint2* rw = reinterpret_cast<const uint2*>(recv);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    // pairs of elements (2j, 2j + 1).  l starts at -0: it stays -0 exactly
    // when every addend is -0 (every code 0x80, since v - h of any other value
    // is +0 or non-zero); an Inf/NaN code makes h or l NaN
    uint64_t h[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      h[j] = f2_pack(0.0f, 0.0f);
      l[j] = f2_pack(-0.0f, -0.0f);
    }
    for (int r0 = 0; r0 < world; r0 += kReduceBatch) {
      // the batch's loads all issue before any of their values is used
      const uint2* p = rw + static_cast<int64_t>(r0) * n8 + i;
      uint2 w[kReduceBatch];
#pragma unroll
      for (int b = 0; b < kReduceBatch; ++b)
        w[b] = r0 + b < world ? __ldcs(p + static_cast<int64_t>(b) * n8) : make_uint2(0u, 0u);
#pragma unroll
      for (int b = 0; b < kReduceBatch; ++b) {
        if (r0 + b >= world) break;
        float2 f[4];
        e5m2x4_values(w[b].x, f[0], f[1]);
        e5m2x4_values(w[b].y, f[2], f[3]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint64_t v = f2_pack(f[j].x, f[j].y);
          const uint64_t hj = f2_add(f2_add(v, up), down);  // nearest integers
          h[j] = f2_add(h[j], hj);
          l[j] = f2_add(l[j], f2_fma(hj, minus1, v));       // v - hj, exact
        }
      }
    }
    uint32_t o[2];
#pragma unroll
    for (int j = 0; j < 4; j += 2)
      o[j >> 1] = e5m2x2_of_exact_sums(h[j], l[j], minus1) | (e5m2x2_of_exact_sums(h[j + 1], l[j + 1], minus1) << 16);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      // a NaN sum (some addend was Inf or NaN) takes the code 0x7E
      // (the conversion saturates, so an exponent field of 31 is a NaN code)
      const uint32_t nan = __vcmpeq4(o[q] & 0x7C7C7C7Cu, 0x7C7C7C7Cu);
      o[q] = (o[q] & ~nan) | (0x7E7E7E7Eu & nan);
    }
    reinterpret_cast<uint2*>(out)[i] = make_uint2(o[0], o[1]);
  }
}

// ---- 6. bf16(fp32(decode(code) * f)) ----------------------------------------
__device__ __forceinline__ float e5m2_value(uint32_t c) {
  // an E5M2 code is the top byte of the binary16 value it encodes
  return __half2float(__ushort_as_half(static_cast<unsigned short>(c << 8)));
}

__global__ void __launch_bounds__(kThreads) grad_dequantize_kernel(const uint8_t* __restrict__ codes, int64_t n,
                                                                   const float* scale, int world, int average,
                                                                   uint16_t* __restrict__ out) {
  const float f = average ? __fdiv_rn(scale[1], static_cast<float>(world)) : scale[1];
  const int64_t n8 = n / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; i < n8; i += 2 * stride) {
    const bool two = i + stride < n8;  // two loads in flight per thread
    const uint2 v0 = reinterpret_cast<const uint2*>(codes)[i];
    const uint2 v1 = two ? reinterpret_cast<const uint2*>(codes)[i + stride] : make_uint2(0u, 0u);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint2 v = h == 0 ? v0 : v1;
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t w = j < 2 ? v.x : v.y;
        const uint32_t lo = (w >> (16 * (j & 1))) & 0xFFu, hi = (w >> (16 * (j & 1) + 8)) & 0xFFu;
        const __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(e5m2_value(lo), f), __fmul_rn(e5m2_value(hi), f));
        o[j] = *reinterpret_cast<const uint32_t*>(&b);
      }
      if (h == 0 || two) reinterpret_cast<uint4*>(out)[i + h * stride] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  for (int64_t i = 8 * n8 + blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; i < n; i += stride) {
    const __nv_bfloat16 b = __float2bfloat16_rn(__fmul_rn(e5m2_value(codes[i]), f));
    out[i] = *reinterpret_cast<const uint16_t*>(&b);
  }
}

int grid_for(int64_t units, int num_sms) {
  const int64_t blocks = (units + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  return static_cast<int>(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

}  // namespace

cudaError_t launch_grad_amax(const void* g, int64_t n, float* amax, int num_sms, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), s);
  if (e != cudaSuccess) return e;
  grad_amax_kernel<<<one_pass_grid(n / 8), kThreads, 0, s>>>(static_cast<const uint16_t*>(g), n,
                                                              reinterpret_cast<uint32_t*>(amax));
  return cudaGetLastError();
}

cudaError_t launch_grad_quantize(const void* g, int64_t n, const float* amax, int world, void* codes,
                                 int64_t padded_n, float* scale, int num_sms, cudaStream_t s) {
  grad_quantize_kernel<<<one_pass_grid(padded_n / 8), kThreads, 0, s>>>(
      static_cast<const uint16_t*>(g), n, amax, world, static_cast<uint8_t*>(codes), padded_n, scale);
  return cudaGetLastError();
}

cudaError_t launch_grad_reduce(const void* recv, int world, int64_t chunk, void* out, int num_sms, cudaStream_t s) {
  if (world <= kReduceF32MaxWorld)
    grad_reduce_f32_kernel<<<std::min(grid_for(chunk / 8, num_sms), kReduceCtasPerSm * num_sms), kThreads, 0, s>>>(
        static_cast<const uint8_t*>(recv), world, chunk, static_cast<uint8_t*>(out));
  else
    grad_reduce_kernel<<<grid_for(chunk / 4, num_sms), kThreads, 0, s>>>(static_cast<const uint8_t*>(recv), world,
                                                                         chunk, static_cast<uint8_t*>(out));
  return cudaGetLastError();
}

cudaError_t launch_grad_dequantize(const void* codes, int64_t n, const float* scale, int world, int average,
                                   void* out, int num_sms, cudaStream_t s) {
  grad_dequantize_kernel<<<grid_for(n / 8 + 1, num_sms), kThreads, 0, s>>>(
      static_cast<const uint8_t*>(codes), n, scale, world, average, static_cast<uint16_t*>(out));
  return cudaGetLastError();
}

}  // namespace fp8lin
