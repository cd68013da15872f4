// cast_kernels.cu -- amax + scale + saturating FP8 cast, and the end-of-step
// scale update ("4.2 Hopper I -- Transformer Engine / FP8", S4.2.4 and S4.2.6).
//
// Kernels (all HBM-bound; see each for its bytes per element):
//  * amax_cast_flat      one pass over a bf16 tensor: 16-byte loads, |x| max,
//                        x*scale -> cvt.rn.satfinite to E4M3/E5M2, 16-byte stores,
//                        saturation/underflow counts; the block that finishes
//                        last folds the tensor's amax into its state and, when
//                        asked, rolls the history and sets the next scale.
//  * amax_cast_transpose the same on a 2-D tensor, tiled 128x128 through shared
//                        memory, also writing the transposed codes.
//  * amax_only           the first pass of current scaling (amax only).
//  * update_scales       end of step: roll every recorded tensor's history.
#include <cfloat>
#include <cstdint>

#include "state.cuh"

namespace fp8lin {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 128;  // cast-transpose tile edge (elements)

template <int FMT>
__device__ __forceinline__ float fp8_max() {
  return FMT == kE4M3 ? kMaxE4M3 : kMaxE5M2;
}

// Two fp32 -> two FP8 codes, round to nearest even, saturating to +-FP8_MAX
// (NaN stays NaN).  Result: lo in bits 0-7, hi in bits 8-15.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_pair(float lo, float hi) {
  unsigned short r;
  if (FMT == kE4M3)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(uint4* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Per-thread partial results.  Underflow = (#zero codes) - (#zero inputs): a
// zero input always gives a zero code, so the difference counts exactly the
// nonzero inputs that were flushed to +-0.  Zeros are counted with SIMD
// compares: 8 set bits per zero byte, 16 per zero bf16.
struct Acc {
  uint32_t amax2;   // two packed 16-bit maxima of |bf16| bit patterns
  uint32_t sat;
  uint32_t zq_bits;
  uint32_t zx_bits;
  uint32_t und_direct;  // underflows counted element by element (edges)
};

// 8 bf16 -> 8 codes.
template <int FMT>
__device__ __forceinline__ uint2 cast8(uint4 v, float s, Acc& a) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o0 = 0, o1 = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t mag = w[j] & 0x7FFF7FFFu;
    a.amax2 = __vmaxu2(a.amax2, mag);
    a.zx_bits += __popc(__vcmpeq2(mag, 0u));
    const float lo = __uint_as_float(w[j] << 16);
    const float hi = __uint_as_float(w[j] & 0xFFFF0000u);
    const float plo = __fmul_rn(lo, s);
    const float phi = __fmul_rn(hi, s);
    a.sat += (fabsf(plo) > fp8_max<FMT>()) + (fabsf(phi) > fp8_max<FMT>());
    const uint32_t p = cvt_pair<FMT>(plo, phi);
    if (j == 0) o0 = p;
    else if (j == 1) o0 |= p << 16;
    else if (j == 2) o1 = p;
    else o1 |= p << 16;
  }
  a.zq_bits += __popc(__vcmpeq4(o0 & 0x7F7F7F7Fu, 0u)) + __popc(__vcmpeq4(o1 & 0x7F7F7F7Fu, 0u));
  return make_uint2(o0, o1);
}

// One element (edges and tails).
template <int FMT>
__device__ __forceinline__ uint8_t cast1(uint16_t b, float s, Acc& a) {
  const uint32_t mag = b & 0x7FFFu;
  a.amax2 = __vmaxu2(a.amax2, mag);
  const float p = __fmul_rn(__uint_as_float((uint32_t)b << 16), s);
  a.sat += fabsf(p) > fp8_max<FMT>();
  const uint32_t c = cvt_pair<FMT>(p, 0.0f) & 0xFFu;
  a.und_direct += (mag != 0u) && ((c & 0x7Fu) == 0u);
  return (uint8_t)c;
}

// scale = FP8_MAX / m in fp32; keep `prev` when m is 0, NaN or Inf; clamp an
// overflowing quotient to FLT_MAX.
template <int FMT>
__device__ __forceinline__ float scale_from_amax(float m, float prev) {
  if (!(m > 0.0f) || !(m <= FLT_MAX)) return prev;
  float s = __fdiv_rn(fp8_max<FMT>(), m);
  return s > FLT_MAX ? FLT_MAX : s;
}

// The scale a cast uses: the stored delayed scale, or (current scaling) the
// one derived from the amax the first pass left in amax_acc.
template <int FMT, bool CURRENT>
__device__ __forceinline__ void cast_scale(const TensorState* st, float& s, float& sinv) {
  if (CURRENT) {
    const uint32_t ab = *reinterpret_cast<const volatile uint32_t*>(&st->amax_acc);
    s = scale_from_amax<FMT>(__uint_as_float(ab), st->scale);
    sinv = __frcp_rn(s);
  } else {
    s = st->scale;
    sinv = st->scale_inv;
  }
}

// Push the pending amax into the ring and derive the next scale (S4.2.4's
// delayed scaling; S4.2.6's history length and "max" rule).
__device__ void roll_and_rescale(TensorState* st, float* h, int H, int algo) {
  const uint32_t a = st->amax_pending;
  int head = st->head + 1;
  if (head >= H) head = 0;
  st->head = head;
  h[head] = __uint_as_float(a);
  uint32_t m = a;
  if (algo == 0) {
    m = 0u;
    for (int i = 0; i < H; ++i) m = max(m, __float_as_uint(h[i]));
  }
  const float mf = __uint_as_float(m);
  if (mf > 0.0f && mf <= FLT_MAX) {
    const float fmax = st->dtype == kE5M2 ? kMaxE5M2 : kMaxE4M3;
    float s = __fdiv_rn(fmax, mf);
    if (s > FLT_MAX) s = FLT_MAX;
    st->scale = s;
    st->scale_inv = __frcp_rn(s);
  }
  st->amax_last = a;
  st->n_sat_last = st->n_sat;
  st->n_und_last = st->n_und;
  st->amax_pending = 0u;
  st->n_sat = 0ull;
  st->n_und = 0ull;
  st->recorded = 0;
}

// Block reduction of the partials, atomics into the tensor state, and the
// last-block tail that closes the cast.
template <int FMT>
__device__ void block_finish(const Acc& a, bool record_amax, TensorState* st, float* hist, int H,
                             int algo, int update_now, float s, float sinv) {
  __shared__ uint32_t sh_amax[kThreads / 32];
  __shared__ uint32_t sh_sat[kThreads / 32];
  __shared__ uint32_t sh_und[kThreads / 32];
  __shared__ int sh_last;
  const uint32_t amax_bits = max(a.amax2 & 0xFFFFu, a.amax2 >> 16) << 16;
  const uint32_t und = a.zq_bits / 8u - a.zx_bits / 16u + a.und_direct;
  const uint32_t wa = __reduce_max_sync(0xFFFFFFFFu, amax_bits);
  const uint32_t ws = __reduce_add_sync(0xFFFFFFFFu, a.sat);
  const uint32_t wu = __reduce_add_sync(0xFFFFFFFFu, und);
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    sh_amax[warp] = wa;
    sh_sat[warp] = ws;
    sh_und[warp] = wu;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t am = 0u;
    unsigned long long bs = 0ull, bu = 0ull;
    for (int i = 0; i < kThreads / 32; ++i) {
      am = max(am, sh_amax[i]);
      bs += sh_sat[i];
      bu += sh_und[i];
    }
    if (record_amax && am) atomicMax(&st->amax_acc, am);
    if (bs) atomicAdd(&st->sat_acc, bs);
    if (bu) atomicAdd(&st->und_acc, bu);
    __threadfence();
    const uint32_t t = atomicAdd(&st->ticket, 1u);
    sh_last = (t == gridDim.x - 1);
  }
  __syncthreads();
  if (sh_last && threadIdx.x == 0) {
    __threadfence();
    const uint32_t am = atomicExch(&st->amax_acc, 0u);
    const unsigned long long ns = atomicExch(&st->sat_acc, 0ull);
    const unsigned long long nu = atomicExch(&st->und_acc, 0ull);
    atomicExch(&st->ticket, 0u);
    st->amax_pending = max(st->amax_pending, am);
    st->n_sat += ns;
    st->n_und += nu;
    st->recorded = 1;
    st->cast_scale = s;
    st->cast_scale_inv = sinv;
    st->dtype = FMT;
    if (update_now) roll_and_rescale(st, hist, H, algo);
    __threadfence();
  }
}

// ---------------------------------------------------------------------------
// Flat one-pass cast.  Algorithmic traffic: 2 B read + 1 B written per element.
// ---------------------------------------------------------------------------
template <int FMT, bool CURRENT>
__global__ void __launch_bounds__(kThreads) amax_cast_flat(const uint4* __restrict__ x,
                                                           uint4* __restrict__ q, int64_t n,
                                                           TensorState* st, float* hist, int H,
                                                           int algo, int update_now) {
  float s, sinv;
  cast_scale<FMT, CURRENT>(st, s, sinv);
  Acc a{0u, 0u, 0u, 0u, 0u};
  const int64_t nv = n >> 4;  // 16-element units: 32 B in, 16 B out
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + stride < nv; i += 2 * stride) {
    const uint4 v0 = ld_stream(x + 2 * i);
    const uint4 v1 = ld_stream(x + 2 * i + 1);
    const uint4 v2 = ld_stream(x + 2 * (i + stride));
    const uint4 v3 = ld_stream(x + 2 * (i + stride) + 1);
    const uint2 c0 = cast8<FMT>(v0, s, a);
    const uint2 c1 = cast8<FMT>(v1, s, a);
    const uint2 c2 = cast8<FMT>(v2, s, a);
    const uint2 c3 = cast8<FMT>(v3, s, a);
    st_stream(q + i, make_uint4(c0.x, c0.y, c1.x, c1.y));
    st_stream(q + i + stride, make_uint4(c2.x, c2.y, c3.x, c3.y));
  }
  if (i < nv) {
    const uint4 v0 = ld_stream(x + 2 * i);
    const uint4 v1 = ld_stream(x + 2 * i + 1);
    const uint2 c0 = cast8<FMT>(v0, s, a);
    const uint2 c1 = cast8<FMT>(v1, s, a);
    st_stream(q + i, make_uint4(c0.x, c0.y, c1.x, c1.y));
  }
  if (blockIdx.x == gridDim.x - 1) {  // the < 16 trailing elements
    const int64_t e = nv * 16 + threadIdx.x;
    if (e < n) {
      const uint16_t b = reinterpret_cast<const uint16_t*>(x)[e];
      reinterpret_cast<uint8_t*>(q)[e] = cast1<FMT>(b, s, a);
    }
  }
  block_finish<FMT>(a, !CURRENT, st, hist, H, algo, update_now, s, sinv);
}

// ---------------------------------------------------------------------------
// Cast + transpose of a [rows, cols] tensor.  Algorithmic traffic: 2 B read,
// 1 B q and 1 B q^T written per element.  128x128 tiles staged in shared
// memory as 32-bit words whose column index is XOR-swizzled by the row's
// 16-row group, so the transposing reads (16 rows x 4 bytes per thread) hit 32
// distinct banks.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int swz(int lr, int word) {
  return lr * 32 + (word ^ (((lr >> 4) & 7) << 2));
}

template <int FMT, bool CURRENT>
__global__ void __launch_bounds__(kThreads) amax_cast_transpose(
    const uint16_t* __restrict__ x, uint8_t* __restrict__ q, uint8_t* __restrict__ qt,
    int64_t rows, int64_t cols, TensorState* st, float* hist, int H, int algo, int update_now) {
  __shared__ __align__(16) uint32_t tile[kTile * kTile / 4];
  float s, sinv;
  cast_scale<FMT, CURRENT>(st, s, sinv);
  Acc a{0u, 0u, 0u, 0u, 0u};
  const int64_t tiles_c = (cols + kTile - 1) / kTile;
  const int64_t tiles = ((rows + kTile - 1) / kTile) * tiles_c;
  const bool vec_cols = (cols % 16) == 0;
  const bool vec_rows = (rows % 16) == 0;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int64_t r0 = (t / tiles_c) * kTile;
    const int64_t c0 = (t % tiles_c) * kTile;
    // phase 1: cast 16-element row chunks, write q, stash codes
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int u = threadIdx.x + it * kThreads;
      const int lr = u >> 3;
      const int ch = u & 7;
      const int64_t r = r0 + lr;
      const int64_t c = c0 + ch * 16;
      uint4 codes;
      if (vec_cols && r < rows && c + 16 <= cols) {
        const uint4* src = reinterpret_cast<const uint4*>(x + r * cols + c);
        const uint4 v0 = ld_stream(src);
        const uint4 v1 = ld_stream(src + 1);
        const uint2 c01 = cast8<FMT>(v0, s, a);
        const uint2 c23 = cast8<FMT>(v1, s, a);
        codes = make_uint4(c01.x, c01.y, c23.x, c23.y);
        *reinterpret_cast<uint4*>(q + r * cols + c) = codes;
      } else {
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        for (int e = 0; e < 16; ++e) {
          if (r < rows && c + e < cols) {
            const uint8_t code = cast1<FMT>(x[r * cols + c + e], s, a);
            q[r * cols + c + e] = code;
            w[e >> 2] |= (uint32_t)code << (8 * (e & 3));
          }
        }
        codes = make_uint4(w[0], w[1], w[2], w[3]);
      }
      *reinterpret_cast<uint4*>(&tile[swz(lr, ch * 4)]) = codes;
    }
    __syncthreads();
    // phase 2: lane -> (h: 16-row group, g: 4-column group); a warp writes
    // 4 columns x 128 rows = four full 128-byte lines of q^T.
    {
      const int h = lane & 7;
      const int g = (lane >> 3) + 4 * warp;
      uint32_t out[4][4];  // [column j][row block b]
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int lr = 16 * h + 4 * b;
        const uint32_t w0 = tile[swz(lr + 0, g)];
        const uint32_t w1 = tile[swz(lr + 1, g)];
        const uint32_t w2 = tile[swz(lr + 2, g)];
        const uint32_t w3 = tile[swz(lr + 3, g)];
        const uint32_t t0 = __byte_perm(w0, w1, 0x5140);
        const uint32_t t1 = __byte_perm(w2, w3, 0x5140);
        const uint32_t t2 = __byte_perm(w0, w1, 0x7362);
        const uint32_t t3 = __byte_perm(w2, w3, 0x7362);
        out[0][b] = __byte_perm(t0, t1, 0x5410);
        out[1][b] = __byte_perm(t0, t1, 0x7632);
        out[2][b] = __byte_perm(t2, t3, 0x5410);
        out[3][b] = __byte_perm(t2, t3, 0x7632);
      }
      const int64_t rs = r0 + 16 * h;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t col = c0 + 4 * g + j;
        if (col >= cols) continue;
        uint8_t* dst = qt + col * rows + rs;
        if (vec_rows && rs + 16 <= rows) {
          *reinterpret_cast<uint4*>(dst) = make_uint4(out[j][0], out[j][1], out[j][2], out[j][3]);
        } else {
          for (int e = 0; e < 16; ++e)
            if (rs + e < rows) dst[e] = (uint8_t)(out[j][e >> 2] >> (8 * (e & 3)));
        }
      }
    }
    __syncthreads();
  }
  block_finish<FMT>(a, !CURRENT, st, hist, H, algo, update_now, s, sinv);
}

// ---------------------------------------------------------------------------
// First pass of current scaling: amax only (2 B read per element).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) amax_only(const uint4* __restrict__ x, int64_t n,
                                                      TensorState* st) {
  uint32_t m2 = 0u;
  const int64_t nv = n >> 3;  // 8-element units
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < nv; i += 4 * stride) {
    const uint4 v0 = ld_stream(x + i);
    const uint4 v1 = ld_stream(x + i + stride);
    const uint4 v2 = ld_stream(x + i + 2 * stride);
    const uint4 v3 = ld_stream(x + i + 3 * stride);
    m2 = __vmaxu2(m2, (__vmaxu2(__vmaxu2(v0.x & 0x7FFF7FFFu, v0.y & 0x7FFF7FFFu),
                                __vmaxu2(v0.z & 0x7FFF7FFFu, v0.w & 0x7FFF7FFFu))));
    m2 = __vmaxu2(m2, (__vmaxu2(__vmaxu2(v1.x & 0x7FFF7FFFu, v1.y & 0x7FFF7FFFu),
                                __vmaxu2(v1.z & 0x7FFF7FFFu, v1.w & 0x7FFF7FFFu))));
    m2 = __vmaxu2(m2, (__vmaxu2(__vmaxu2(v2.x & 0x7FFF7FFFu, v2.y & 0x7FFF7FFFu),
                                __vmaxu2(v2.z & 0x7FFF7FFFu, v2.w & 0x7FFF7FFFu))));
    m2 = __vmaxu2(m2, (__vmaxu2(__vmaxu2(v3.x & 0x7FFF7FFFu, v3.y & 0x7FFF7FFFu),
                                __vmaxu2(v3.z & 0x7FFF7FFFu, v3.w & 0x7FFF7FFFu))));
  }
  for (; i < nv; i += stride) {
    const uint4 v = ld_stream(x + i);
    m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                               __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
  }
  if (blockIdx.x == gridDim.x - 1) {
    const int64_t e = nv * 8 + threadIdx.x;
    if (e < n) m2 = __vmaxu2(m2, reinterpret_cast<const uint16_t*>(x)[e] & 0x7FFFu);
  }
  uint32_t am = max(m2 & 0xFFFFu, m2 >> 16) << 16;
  am = __reduce_max_sync(0xFFFFFFFFu, am);
  __shared__ uint32_t sh[kThreads / 32];
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = am;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t b = 0u;
    for (int k = 0; k < kThreads / 32; ++k) b = max(b, sh[k]);
    if (b) atomicMax(&st->amax_acc, b);
  }
}

__global__ void update_scales_kernel(TensorState* states, float* hist, int T, int H, int algo) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  TensorState* st = states + t;
  if (!st->recorded) return;
  roll_and_rescale(st, hist + (int64_t)t * H, H, algo);
}

// history_in: H values, oldest first (already validated: finite or NaN, >= +0).
__global__ void set_state_kernel(TensorState* st, float* h, const float* history_in, int H,
                                 float scale, int dtype) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  for (int i = 0; i < H; ++i) h[i] = history_in[i];
  st->head = H - 1;
  st->scale = scale;
  st->scale_inv = __frcp_rn(scale);
  st->cast_scale = scale;
  st->cast_scale_inv = st->scale_inv;
  st->amax_acc = 0u;
  st->amax_pending = 0u;
  st->ticket = 0u;
  st->sat_acc = st->und_acc = 0ull;
  st->n_sat = st->n_und = 0ull;
  st->recorded = 0;
  st->dtype = dtype;
}

template <typename K>
int blocks_per_sm(K kernel) {
  int b = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kThreads, 0) != cudaSuccess || b < 1)
    b = 1;
  return b;
}

template <int FMT, bool CURRENT>
cudaError_t launch_cast_t(const RecipeDev& rd, int id, const void* x, int64_t rows, int64_t cols,
                          bool update_now, void* out, void* out_t, int num_sms, cudaStream_t s) {
  TensorState* st = rd.states + id;
  float* h = rd.history + (int64_t)id * rd.H;
  const int64_t n = rows * cols;
  if (CURRENT) {
    static const int bpa = blocks_per_sm(amax_only);
    const int64_t units = (n + 7) / 8;
    int64_t grid = (units + kThreads - 1) / kThreads;
    if (grid > (int64_t)num_sms * bpa) grid = (int64_t)num_sms * bpa;
    if (grid < 1) grid = 1;
    amax_only<<<(unsigned)grid, kThreads, 0, s>>>(static_cast<const uint4*>(x), n, st);
  }
  if (out_t == nullptr) {
    static const int bp = blocks_per_sm(amax_cast_flat<FMT, CURRENT>);
    const int64_t units = (n + 15) / 16;
    int64_t grid = (units + kThreads - 1) / kThreads;
    if (grid > (int64_t)num_sms * bp) grid = (int64_t)num_sms * bp;
    if (grid < 1) grid = 1;
    amax_cast_flat<FMT, CURRENT><<<(unsigned)grid, kThreads, 0, s>>>(
        static_cast<const uint4*>(x), static_cast<uint4*>(out), n, st, h, rd.H, rd.algo,
        update_now ? 1 : 0);
  } else {
    static const int bp = blocks_per_sm(amax_cast_transpose<FMT, CURRENT>);
    const int64_t tiles = ((rows + kTile - 1) / kTile) * ((cols + kTile - 1) / kTile);
    int64_t grid = tiles;
    if (grid > (int64_t)num_sms * bp) grid = (int64_t)num_sms * bp;
    amax_cast_transpose<FMT, CURRENT><<<(unsigned)grid, kThreads, 0, s>>>(
        static_cast<const uint16_t*>(x), static_cast<uint8_t*>(out), static_cast<uint8_t*>(out_t),
        rows, cols, st, h, rd.H, rd.algo, update_now ? 1 : 0);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_amax_cast(const RecipeDev& rd, int tensor_id, const void* x, int64_t rows,
                             int64_t cols, int dtype, bool current, bool update_now, void* out,
                             void* out_t, int num_sms, cudaStream_t s) {
  if (dtype == kE4M3) {
    return current ? launch_cast_t<kE4M3, true>(rd, tensor_id, x, rows, cols, update_now, out, out_t, num_sms, s)
                   : launch_cast_t<kE4M3, false>(rd, tensor_id, x, rows, cols, update_now, out, out_t, num_sms, s);
  }
  return current ? launch_cast_t<kE5M2, true>(rd, tensor_id, x, rows, cols, update_now, out, out_t, num_sms, s)
                 : launch_cast_t<kE5M2, false>(rd, tensor_id, x, rows, cols, update_now, out, out_t, num_sms, s);
}

cudaError_t launch_update_scales(const RecipeDev& rd, cudaStream_t s) {
  const int threads = 128;
  const int grid = (rd.num_tensors + threads - 1) / threads;
  update_scales_kernel<<<grid, threads, 0, s>>>(rd.states, rd.history, rd.num_tensors, rd.H, rd.algo);
  return cudaGetLastError();
}

cudaError_t launch_set_state(const RecipeDev& rd, int tensor_id, const float* history_dev,
                             float scale, int dtype, cudaStream_t s) {
  set_state_kernel<<<1, 32, 0, s>>>(rd.states + tensor_id, rd.history + (int64_t)tensor_id * rd.H,
                                    history_dev, rd.H, scale, dtype);
  return cudaGetLastError();
}

}  // namespace fp8lin
