// noalloc_cast.cu -- a current-scaling FP8 cast that allocates no device memory.
//
// Some callers cannot call cudaMalloc: code that runs inside a host framework
// which owns all device memory and forbids allocation while it executes (for
// example a plugin's enqueue step, or a runtime with a fixed memory plan), and
// code that must not risk the device-wide synchronisation an allocation can
// cause.  fp8_quantize_current_noalloc serves them: the caller passes only the
// input and the outputs, and the cross-block scratch of the two passes (one
// amax per block, one pair of counts per block, two completion tickets) lives in
// a file-scope __device__ array that is part of the loaded library.
//
// That array is one per GPU that loads the library, held until the process
// exits, and shared by every call on that GPU: calls that overlap on the GPU
// (different streams, no ordering between them) race on it.  Its host-side
// name is not a device address; the device address is looked up once per
// device with cudaGetSymbolAddress, by the first call made on that device
// (make that first call before any stream capture).  The address kept is the
// one in the device's primary context; it is not refreshed after
// cudaDeviceReset.
#include <cfloat>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "fp8lin.h"
#include "state.cuh"
#include "tc_ptx.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int64_t kChunk = 65536;    // elements per block; a block's counts fit in 32 bits
constexpr int kMaxBlocks = 16384;    // scratch slots
constexpr int kMaxDevices = 64;

struct Scratch {
  unsigned int ticket_amax;  // blocks finished in pass 1 (cleared before each call)
  unsigned int ticket_cast;  // blocks finished in pass 2 (cleared before each call)
  float scale;               // written by pass 1's last block
  float scale_inv;
  unsigned int pad[60];
  unsigned int part_amax[kMaxBlocks];  // fp32 bit patterns of per-block max|x|
  unsigned int part_sat[kMaxBlocks];
  unsigned int part_und[kMaxBlocks];
};
static_assert(FP8_NOALLOC_MAX_ELEMENTS == kChunk * kMaxBlocks, "limit and scratch size disagree");

static __device__ __align__(256) Scratch g_scratch;

template <int FMT>
__device__ __forceinline__ float fmax_of() {
  return FMT == 0 ? 448.0f : 57344.0f;
}

// Pass 1: per-block max|x| into scratch; the last block reduces them and sets
// scale = FP8_MAX / amax (kept at 1 when amax is 0 or not finite; an
// overflowing quotient is clamped to FLT_MAX) and scale_inv = 1/scale.
template <int FMT>
__global__ void __launch_bounds__(kThreads) noalloc_amax(const uint16_t* __restrict__ x, int64_t n,
                                                         Scratch* sc, float* scale_out) {
  const int64_t begin = (int64_t)blockIdx.x * kChunk;
  const int64_t end = begin + kChunk < n ? begin + kChunk : n;
  unsigned int m2 = 0u;
  const bool vec = ((end - begin) & 7) == 0;
  if (vec) {
    const uint4* v = reinterpret_cast<const uint4*>(x + begin);
    const int64_t nv = (end - begin) >> 3;
    for (int64_t i = threadIdx.x; i < nv; i += kThreads) {
      const uint4 w = v[i];
      m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu),
                                 __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu)));
    }
  } else {
    for (int64_t i = begin + threadIdx.x; i < end; i += kThreads) m2 = __vmaxu2(m2, x[i] & 0x7FFFu);
  }
  unsigned int am = max(m2 & 0xFFFFu, m2 >> 16) << 16;
  am = __reduce_max_sync(0xFFFFFFFFu, am);
  __shared__ unsigned int sh[kThreads / 32];
  __shared__ int last;
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = am;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned int b = 0u;
    for (int k = 0; k < kThreads / 32; ++k) b = max(b, sh[k]);
    sc->part_amax[blockIdx.x] = b;
    __threadfence();
    last = atomicAdd(&sc->ticket_amax, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  unsigned int b = 0u;
  for (int i = threadIdx.x; i < (int)gridDim.x; i += kThreads)
    b = max(b, *reinterpret_cast<volatile unsigned int*>(&sc->part_amax[i]));
  b = __reduce_max_sync(0xFFFFFFFFu, b);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = b;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned int a = 0u;
    for (int k = 0; k < kThreads / 32; ++k) a = max(a, sh[k]);
    const float m = __uint_as_float(a);
    float s = 1.0f;
    if (m > 0.0f && m <= FLT_MAX) {
      s = __fdiv_rn(fmax_of<FMT>(), m);
      if (s > FLT_MAX) s = FLT_MAX;
    }
    const float sinv = __frcp_rn(s);
    sc->scale = s;
    sc->scale_inv = sinv;
    scale_out[0] = s;
    scale_out[1] = sinv;
    __threadfence();
  }
}

// Pass 2: cast with the scale pass 1 left in scratch; per-block saturation and
// underflow counts into scratch; the last block sums them into counts_out.
template <int FMT>
__global__ void __launch_bounds__(kThreads) noalloc_cast(const uint16_t* __restrict__ x, int64_t n,
                                                         uint8_t* __restrict__ out, Scratch* sc,
                                                         unsigned long long* counts_out) {
  const float s = *reinterpret_cast<volatile float*>(&sc->scale);
  const int64_t begin = (int64_t)blockIdx.x * kChunk;
  const int64_t end = begin + kChunk < n ? begin + kChunk : n;
  unsigned int sat = 0u, und = 0u;
  const bool vec = ((end - begin) & 15) == 0;
  if (vec) {
    const uint4* v = reinterpret_cast<const uint4*>(x + begin);
    uint4* o = reinterpret_cast<uint4*>(out + begin);
    const int64_t nv = (end - begin) >> 4;
    for (int64_t i = threadIdx.x; i < nv; i += kThreads) {
      const uint4 a = v[2 * i];
      const uint4 b = v[2 * i + 1];
      const unsigned int w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      unsigned int c[4];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float lo = __uint_as_float(w[j] << 16);
        const float hi = __uint_as_float(w[j] & 0xFFFF0000u);
        const float plo = __fmul_rn(lo, s);
        const float phi = __fmul_rn(hi, s);
        sat += (fabsf(plo) > fmax_of<FMT>()) + (fabsf(phi) > fmax_of<FMT>());
        const unsigned int p = fp8lin::cvt_fp8x2<FMT>(plo, phi);
        und += ((w[j] & 0x7FFFu) != 0u && (p & 0x7Fu) == 0u) +
               ((w[j] & 0x7FFF0000u) != 0u && (p & 0x7F00u) == 0u);
        if (j & 1) c[j >> 1] |= p << 16;
        else c[j >> 1] = p;
      }
      o[i] = make_uint4(c[0], c[1], c[2], c[3]);
    }
  } else {
    for (int64_t i = begin + threadIdx.x; i < end; i += kThreads) {
      const unsigned int b = x[i];
      const float p = __fmul_rn(__uint_as_float(b << 16), s);
      sat += fabsf(p) > fmax_of<FMT>();
      const unsigned int c = fp8lin::cvt_fp8x2<FMT>(p, 0.0f) & 0xFFu;
      und += (b & 0x7FFFu) != 0u && (c & 0x7Fu) == 0u;
      out[i] = (uint8_t)c;
    }
  }
  sat = __reduce_add_sync(0xFFFFFFFFu, sat);
  und = __reduce_add_sync(0xFFFFFFFFu, und);
  __shared__ unsigned int sh_s[kThreads / 32], sh_u[kThreads / 32];
  __shared__ int last;
  if ((threadIdx.x & 31) == 0) {
    sh_s[threadIdx.x >> 5] = sat;
    sh_u[threadIdx.x >> 5] = und;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned int bs = 0u, bu = 0u;
    for (int k = 0; k < kThreads / 32; ++k) {
      bs += sh_s[k];
      bu += sh_u[k];
    }
    sc->part_sat[blockIdx.x] = bs;
    sc->part_und[blockIdx.x] = bu;
    __threadfence();
    last = atomicAdd(&sc->ticket_cast, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!last || counts_out == nullptr) return;
  __threadfence();
  __shared__ unsigned long long tot_s[kThreads / 32], tot_u[kThreads / 32];
  unsigned long long ts = 0ull, tu = 0ull;
  for (int i = threadIdx.x; i < (int)gridDim.x; i += kThreads) {
    ts += *reinterpret_cast<volatile unsigned int*>(&sc->part_sat[i]);
    tu += *reinterpret_cast<volatile unsigned int*>(&sc->part_und[i]);
  }
  for (int off = 16; off > 0; off >>= 1) {
    ts += __shfl_down_sync(0xFFFFFFFFu, ts, off);
    tu += __shfl_down_sync(0xFFFFFFFFu, tu, off);
  }
  if ((threadIdx.x & 31) == 0) {
    tot_s[threadIdx.x >> 5] = ts;
    tot_u[threadIdx.x >> 5] = tu;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long a = 0ull, b = 0ull;
    for (int k = 0; k < kThreads / 32; ++k) {
      a += tot_s[k];
      b += tot_u[k];
    }
    counts_out[0] = a;
    counts_out[1] = b;
  }
}

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

fp8_status_t fail(fp8_status_t st, const char* fmt, ...) {
  char buf[256];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  fp8lin::set_last_error(buf);
  return st;
}

fp8_status_t scratch_for_current_device(Scratch** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail(FP8_ERR_CUDA, "no usable current CUDA device");
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(FP8_ERR_CUDA, "cudaGetSymbolAddress of the scratch array: %s",
                  cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = static_cast<Scratch*>(g_scratch_ptr[dev]);
  return FP8_OK;
}

}  // namespace

extern "C" fp8_status_t fp8_quantize_current_noalloc(const void* x, int64_t n, int32_t dtype,
                                                     void* out, float* scale_out,
                                                     uint64_t* counts_out, fp8_stream_t stream) {
  fp8lin::set_last_error("");
  if (!x || !out || !scale_out) return fail(FP8_ERR_INVALID, "x, out and scale_out must not be NULL");
  if (dtype != FP8_E4M3 && dtype != FP8_E5M2)
    return fail(FP8_ERR_INVALID, "unknown dtype %d", (int)dtype);
  if (n < 1 || n > FP8_NOALLOC_MAX_ELEMENTS)
    return fail(FP8_ERR_INVALID,
                "n = %lld is outside [1, %lld], the size the static scratch array covers",
                (long long)n, (long long)FP8_NOALLOC_MAX_ELEMENTS);
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(out) & 15u))
    return fail(FP8_ERR_INVALID, "x and out must be 16-byte aligned");
  Scratch* sc = nullptr;
  if (fp8_status_t st = scratch_for_current_device(&sc)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the two tickets must start at zero; everything else is written before it is read
  cudaError_t e = cudaMemsetAsync(sc, 0, 2 * sizeof(unsigned int), s);
  const unsigned int blocks = static_cast<unsigned int>((n + kChunk - 1) / kChunk);
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  uint8_t* o = static_cast<uint8_t*>(out);
  unsigned long long* co = reinterpret_cast<unsigned long long*>(counts_out);
  if (e == cudaSuccess) {
    if (dtype == FP8_E4M3) {
      noalloc_amax<0><<<blocks, kThreads, 0, s>>>(xs, n, sc, scale_out);
      noalloc_cast<0><<<blocks, kThreads, 0, s>>>(xs, n, o, sc, co);
    } else {
      noalloc_amax<1><<<blocks, kThreads, 0, s>>>(xs, n, sc, scale_out);
      noalloc_cast<1><<<blocks, kThreads, 0, s>>>(xs, n, o, sc, co);
    }
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return fail(FP8_ERR_CUDA, "noalloc cast launch: %s", cudaGetErrorString(e));
  return FP8_OK;
}
