// cast_kernels.cu -- amax + scale + saturating FP8 cast, and the end-of-step
// scale update ("4.2 Hopper I -- Transformer Engine / FP8", S4.2.4 and S4.2.6).
//
// Kernels (all HBM-bound; see each for its bytes per element):
//  * amax_cast_flat           one pass over a bf16 tensor: every thread loads its
//                             eight 16-byte vectors at once, then |x| max,
//                             x*scale -> cvt.rn.satfinite to E4M3/E5M2, 8-byte
//                             coalesced stores, saturation/underflow counts,
//                             folded by every block into the tensor's state
//                             (no block waits for another); with update_now a
//                             one-thread launch then rolls the history and sets
//                             the next scale.
//  * amax_cast_transpose_tma  the same on a 2-D tensor: 128x128 bf16 tiles
//                             loaded by TMA into a 2-stage ring, codes staged in
//                             shared memory and written both row-major and
//                             transposed (the K-major operands of the backward
//                             GEMMs).
//  * amax_cast_transpose      register-path version for row pitches TMA cannot
//                             describe (cols not a multiple of 8).
//  * amax_only                the first pass of current scaling (amax only), the
//                             same one-pass shape.
//  * update_scales            end of step: roll every recorded tensor's history.
// The TMA cast-transpose bounds every wait on its tile ring (about 1 s); on
// expiry the block sets an error bit in the recipe and stops streaming.  The
// flat kernels have no waits.
#include <algorithm>
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cfloat>
#include <cstdint>
#include <mutex>

#include "state.cuh"
#include "tc_ptx.cuh"

namespace fp8lin {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 128;  // cast-transpose tile edge (elements)

// Flat kernels: each thread loads kFlatU 16-byte vectors (8 bf16 each) before
// using any, so a block covers kThreads * kFlatU * 8 elements in one pass.
constexpr int kFlatU = 8;
constexpr int kFlatBlockVecs = kThreads * kFlatU;  // 16-byte vectors per block

constexpr int kTStages = 2;
constexpr int kTTileBytes = kTile * kTile * 2;   // one bf16 tile
constexpr int kTSmem = kTStages * kTTileBytes + kTile * kTile + 64 + 128;  // + alignment slack

constexpr unsigned long long kCastTimeoutNs = 1000000000ull;

template <int FMT>
__device__ __forceinline__ float underflow_max() {
  // |p| at or below half the smallest subnormal rounds to +-0 (the tie goes to
  // the even code 0): 2^-10 for E4M3, 2^-17 for E5M2.
  return FMT == kE4M3 ? 0.0009765625f : 7.62939453125e-06f;
}

template <int FMT>
__device__ __forceinline__ float fp8_max() {
  return FMT == kE4M3 ? kMaxE4M3 : kMaxE5M2;
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Per-thread partial results.  Saturated: |x*s| > FP8_MAX.  Underflowed: x != 0
// and |x*s| <= half the smallest subnormal (exactly the products that round to
// +-0).  Both are fp32 compares on the product the cast rounds.
struct Acc {
  uint32_t amax2;   // two packed 16-bit maxima of |bf16| bit patterns
  uint32_t sat;
  uint32_t und;
};

// 8 bf16 -> 8 codes.  The counts take a fast path: saturated and underflowed
// products are rare, so the eight products are first tested together -- the
// largest |p| against FP8_MAX and the smallest against the underflow bound
// (NaN drops out of both, as it fails both per-element tests) -- and counted one
// by one only when the group may hold one.
template <int FMT>
__device__ __forceinline__ uint2 cast8(uint4 v, float s, Acc& a) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[2];
  float x[8], p[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    a.amax2 = __vmaxu2(a.amax2, w[j] & 0x7FFF7FFFu);
    x[2 * j] = __uint_as_float(w[j] << 16);
    x[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    p[2 * j] = __fmul_rn(x[2 * j], s);
    p[2 * j + 1] = __fmul_rn(x[2 * j + 1], s);
    const uint32_t c = cvt_fp8x2<FMT>(p[2 * j], p[2 * j + 1]);
    if (j & 1) o[j >> 1] |= c << 16;
    else o[j >> 1] = c;
  }
  float hi = fabsf(p[0]), lo = fabsf(p[0]);
#pragma unroll
  for (int i = 1; i < 8; ++i) {
    hi = fmaxf(hi, fabsf(p[i]));
    lo = fminf(lo, fabsf(p[i]));
  }
  if (hi > fp8_max<FMT>()) {
#pragma unroll
    for (int i = 0; i < 8; ++i) a.sat += fabsf(p[i]) > fp8_max<FMT>();
  }
  if (lo <= underflow_max<FMT>()) {
#pragma unroll
    for (int i = 0; i < 8; ++i) a.und += (x[i] != 0.0f && fabsf(p[i]) <= underflow_max<FMT>());
  }
  return make_uint2(o[0], o[1]);
}

// One element (edges and tails).
template <int FMT>
__device__ __forceinline__ uint8_t cast1(uint16_t b, float s, Acc& a) {
  const uint32_t mag = b & 0x7FFFu;
  a.amax2 = __vmaxu2(a.amax2, mag);
  const float p = __fmul_rn(__uint_as_float((uint32_t)b << 16), s);
  a.sat += fabsf(p) > fp8_max<FMT>();
  const uint32_t c = cvt_fp8x2<FMT>(p, 0.0f) & 0xFFu;
  a.und += (mag != 0u) && ((c & 0x7Fu) == 0u);
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
// one derived from the amax the first pass left in amax_acc (its low word).
template <int FMT, bool CURRENT>
__device__ __forceinline__ void cast_scale(const TensorState* st, float& s, float& sinv) {
  if (CURRENT) {
    // read-only path: the first pass finished before this kernel began, and
    // nothing writes the word during it (a load per thread through L2 queued
    // behind the blocks' count atomics on the same line: E4M3 casts, with
    // underflows in every block, ran 1.5x slower)
    const uint32_t ab = static_cast<uint32_t>(__ldg(&st->amax_acc));
    s = scale_from_amax<FMT>(__uint_as_float(ab), st->scale);
    sinv = __frcp_rn(s);
  } else {
    s = st->scale;
    sinv = st->scale_inv;
  }
}

// ---- bulk-copy / TMA helpers: tc_ptx.cuh ----------------------------------
// Bounded wait for the phase `parity` of a copy barrier; every thread of the
// block waits and the block agrees on the outcome (true = data ready).
__device__ __forceinline__ bool bar_wait_block(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = smem_u32(bar);
  bool ok = mbar_try_wait(addr, parity);
  if (!ok) {
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (;;) {
      for (int i = 0; i < 32 && !ok; ++i) ok = mbar_try_wait(addr, parity);
      if (ok) break;
      uint64_t t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > kCastTimeoutNs) break;
    }
  }
  return !__syncthreads_or(!ok);
}

// After a time-out on ring slot `stg` (parity `ph`) for this block's unit `u`
// of `units`: thread 0 waits (bounded) for every copy the block still has in
// flight -- units u, u + grid, ..., one per ring slot -- so that none lands in
// shared memory after the block has left.
__device__ __forceinline__ void drain_in_flight(uint64_t* bar, int stages, int stg, uint32_t ph, int64_t u,
                                                int64_t units) {
  if (threadIdx.x != 0) return;
  for (int k = 0; k < stages; ++k) {
    if (u + static_cast<int64_t>(k) * gridDim.x >= units) break;
    int sl = stg + k;
    uint32_t p = ph;
    if (sl >= stages) {
      sl -= stages;
      p ^= 1u;
    }
    const uint32_t addr = smem_u32(&bar[sl]);
    const uint64_t t0 = gtimer();
    while (!mbar_try_wait(addr, p) && gtimer() - t0 < kCastTimeoutNs) {
    }
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

// Block reduction of the partials and atomics into the tensor state.  Every
// block folds its counts (and, delayed, its amax) straight into the step's
// totals -- max and sum commute -- and block 0 writes the cast record, so no
// block waits for another: the fire-and-forget reductions cost far less than a
// completion ticket, which a one-pass grid of 2^14 blocks would serialise on
// one address.  Current scaling's amax is final before the cast starts (the
// first pass left it in amax_acc), so block 0 folds it and closes the epoch.
// With update_now the launcher runs the history update as a separate launch.
template <int FMT, bool CURRENT>
__device__ void block_finish(const Acc& a, TensorState* st, float s, float sinv) {
  __shared__ uint32_t sh_amax[kThreads / 32];
  __shared__ uint32_t sh_sat[kThreads / 32];
  __shared__ uint32_t sh_und[kThreads / 32];
  const uint32_t amax_bits = max(a.amax2 & 0xFFFFu, a.amax2 >> 16) << 16;
  const uint32_t wa = CURRENT ? 0u : __reduce_max_sync(0xFFFFFFFFu, amax_bits);
  const uint32_t ws = __reduce_add_sync(0xFFFFFFFFu, a.sat);
  const uint32_t wu = __reduce_add_sync(0xFFFFFFFFu, a.und);
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
    if (CURRENT) {
      if (blockIdx.x == 0) {
        atomicMax(&st->amax_pending, static_cast<uint32_t>(st->amax_acc));
        st->epoch += 1u;  // the next first pass tags above this one
      }
    } else if (am) {
      atomicMax(&st->amax_pending, am);
    }
    if (bs) atomicAdd(&st->n_sat, bs);
    if (bu) atomicAdd(&st->n_und, bu);
    if (blockIdx.x == 0) {
      st->recorded = 1;
      st->cast_scale = s;
      st->cast_scale_inv = sinv;
      st->dtype = FMT;
    }
  }
}

// ---------------------------------------------------------------------------
// Flat one-pass cast.  Algorithmic traffic: 2 B read + 1 B written per element.
// The grid covers the tensor once: every thread issues its kFlatU 16-byte
// loads (vectors base, base + kThreads, ...) before it casts any of them, so a
// mid-size tensor is wholly in flight at once; the codes leave as coalesced
// 8-byte stores.  The n % 8 trailing elements go to the last block, one per
// thread.  (Measured back to back on rotating inputs against the earlier
// persistent kernel that streamed 16 KB chunks through a 6-stage bulk-copy
// ring: 2^24 elements 12.7 -> 12.3 us, 2^26 37.5 -> 32.7 us, 2^28 140.4 ->
// 115.2 us.)  Under current scaling the blocks take the tensor from its end:
// the amax pass just read it from the start, so its last part is still in L2.
// ---------------------------------------------------------------------------
template <int FMT, bool CURRENT>
__global__ void __launch_bounds__(kThreads) amax_cast_flat(const uint16_t* __restrict__ x,
                                                           uint8_t* __restrict__ q, int64_t n,
                                                           TensorState* st) {
  griddep_wait();  // launched with programmatic dependent launch: nothing before this
  const int64_t nv = n >> 3;  // whole 8-element vectors
  const int64_t blk = CURRENT ? gridDim.x - 1 - blockIdx.x : blockIdx.x;
  const int64_t base = blk * kFlatBlockVecs + threadIdx.x;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  uint4 v[kFlatU];
#pragma unroll
  for (int u = 0; u < kFlatU; ++u) {
    const int64_t i = base + u * kThreads;
    v[u] = i < nv ? ld_stream(xv + i) : make_uint4(0u, 0u, 0u, 0u);
  }
  float s, sinv;  // read while the loads are in flight
  cast_scale<FMT, CURRENT>(st, s, sinv);
  Acc a{0u, 0u, 0u};
  uint2* qv = reinterpret_cast<uint2*>(q);
#pragma unroll
  for (int u = 0; u < kFlatU; ++u) {
    const int64_t i = base + u * kThreads;
    if (i < nv) __stcs(qv + i, cast8<FMT>(v[u], s, a));
  }
  if (blk == gridDim.x - 1) {  // trailing elements
    const int64_t e = nv * 8 + threadIdx.x;
    if (e < n) q[e] = cast1<FMT>(x[e], s, a);
  }
  block_finish<FMT, CURRENT>(a, st, s, sinv);
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
    int64_t rows, int64_t cols, TensorState* st) {
  griddep_wait();  // launched with programmatic dependent launch: nothing before this
  __shared__ __align__(16) uint32_t tile[kTile * kTile / 4];
  float s, sinv;
  cast_scale<FMT, CURRENT>(st, s, sinv);
  Acc a{0u, 0u, 0u};
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
  block_finish<FMT, CURRENT>(a, st, s, sinv);
}

// ---------------------------------------------------------------------------
// Cast + transpose with TMA tile loads (cols a multiple of 8, so that the bf16
// row pitch is a multiple of 16 bytes).  Algorithmic traffic: 2 B read, 1 B q
// and 1 B q^T written per element.  A 2-stage ring of 128x128 bf16 tiles
// (zero-filled past the edges) lets the next tile load while this one is
// transposed out.  Phase 1: 16 threads per row, 8 elements each (conflict-free
// 16-byte shared loads), codes to q and into the swizzled code tile; phase 2
// as in amax_cast_transpose.
// ---------------------------------------------------------------------------
template <int FMT, bool CURRENT>
__global__ void __launch_bounds__(kThreads) amax_cast_transpose_tma(
    const __grid_constant__ CUtensorMap tmx, uint8_t* __restrict__ q, uint8_t* __restrict__ qt,
    int64_t rows, int64_t cols, TensorState* st, uint32_t* err, uint32_t extra_tx) {
  griddep_wait();  // launched with programmatic dependent launch: nothing before this
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);  // TMA wants 128 B
  uint32_t* tile = reinterpret_cast<uint32_t*>(smem + kTStages * kTTileBytes);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kTStages * kTTileBytes + kTile * kTile);
  float s, sinv;
  cast_scale<FMT, CURRENT>(st, s, sinv);
  Acc a{0u, 0u, 0u};
  const int64_t tiles_c = (cols + kTile - 1) / kTile;
  const int64_t tiles = ((rows + kTile - 1) / kTile) * tiles_c;
  const bool vec_rows = (rows % 16) == 0;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int k = 0; k < kTStages; ++k) mbar_init(&bar[k], 1);
    fence_mbar_init();
  }
  __syncthreads();
  int64_t t = blockIdx.x;
  if (threadIdx.x == 0) {
    for (int k = 0; k < kTStages; ++k) {
      const int64_t tk = t + (int64_t)k * gridDim.x;
      if (tk < tiles) {
        // extra_tx (0 except under fp8_debug_inject_stall) over-states the first
        // stage's bytes: its wait then runs out and the time-out path is taken
        mbar_expect_tx(&bar[k], kTTileBytes + (k == 0 ? extra_tx : 0u));
        tma_load_2d(smem + k * kTTileBytes, &tmx, &bar[k], (int32_t)((tk % tiles_c) * kTile),
                    (int32_t)((tk / tiles_c) * kTile));
      }
    }
  }
  int stg = 0;
  uint32_t ph = 0;
  for (; t < tiles; t += gridDim.x) {
    const int64_t r0 = (t / tiles_c) * kTile;
    const int64_t c0 = (t % tiles_c) * kTile;
    if (!bar_wait_block(&bar[stg], ph)) {
      if (threadIdx.x == 0) atomicOr(err, kErrTimeoutCast);
      drain_in_flight(bar, kTStages, stg, ph, t, tiles);
      break;
    }
    const uint8_t* in = smem + stg * kTTileBytes;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int u = it * kThreads + threadIdx.x;
      const int lr = u >> 4;
      const int ch = u & 15;
      const int64_t r = r0 + lr;
      const int64_t c = c0 + ch * 8;
      uint2 codes = make_uint2(0u, 0u);
      if (r < rows && c < cols) {  // cols % 8 == 0: the 8 elements are all inside
        codes = cast8<FMT>(*reinterpret_cast<const uint4*>(in + lr * (kTile * 2) + ch * 16), s, a);
        *reinterpret_cast<uint2*>(q + r * cols + c) = codes;
      }
      *reinterpret_cast<uint2*>(&tile[swz(lr, ch * 2)]) = codes;
    }
    __syncthreads();  // code tile complete; input stage free
    if (threadIdx.x == 0) {
      const int64_t tn = t + (int64_t)kTStages * gridDim.x;
      if (tn < tiles) {
        mbar_expect_tx(&bar[stg], kTTileBytes);
        tma_load_2d(smem + stg * kTTileBytes, &tmx, &bar[stg], (int32_t)((tn % tiles_c) * kTile),
                    (int32_t)((tn / tiles_c) * kTile));
      }
    }
    {
      const int h = lane & 7;
      const int g = (lane >> 3) + 4 * warp;
      uint32_t out[4][4];
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
    __syncthreads();  // code tile consumed
    if (++stg == kTStages) {
      stg = 0;
      ph ^= 1u;
    }
  }
  block_finish<FMT, CURRENT>(a, st, s, sinv);
}

// ---------------------------------------------------------------------------
// First pass of current scaling: amax only (2 B read per element).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) amax_only(const uint4* __restrict__ x, int64_t n,
                                                      TensorState* st) {
  griddep_wait();  // launched with programmatic dependent launch: nothing before this
  // (read-only path: the epoch changes only in the cast pass, a later kernel)
  const unsigned long long tag = static_cast<unsigned long long>(__ldg(&st->epoch) + 1u) << 32;
  const int64_t nv = n >> 3;  // whole 8-element vectors
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kFlatBlockVecs + threadIdx.x;
  uint4 v[kFlatU];
#pragma unroll
  for (int u = 0; u < kFlatU; ++u) {
    const int64_t i = base + u * kThreads;
    v[u] = i < nv ? ld_stream(x + i) : make_uint4(0u, 0u, 0u, 0u);
  }
  uint32_t m2 = 0u;
#pragma unroll
  for (int u = 0; u < kFlatU; ++u)
    m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(v[u].x & 0x7FFF7FFFu, v[u].y & 0x7FFF7FFFu),
                               __vmaxu2(v[u].z & 0x7FFF7FFFu, v[u].w & 0x7FFF7FFFu)));
  if (blockIdx.x == gridDim.x - 1) {  // trailing elements
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
    if (b || blockIdx.x == 0) atomicMax(&st->amax_acc, tag | b);  // block 0 opens the epoch
  }
}

__global__ void update_scales_kernel(TensorState* states, float* hist, int T, int H, int algo) {
  griddep_wait();  // launched with programmatic dependent launch: nothing before this
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
  st->amax_acc = 0ull;
  st->epoch = 0u;
  st->amax_pending = 0u;
  st->n_sat = st->n_und = 0ull;
  st->recorded = 0;
  st->dtype = dtype;
}

// Resident blocks per SM of a cast kernel on the current device, after its
// shared-memory opt-in (both per device, taken on the device's first launch).
template <typename K>
cudaError_t blocks_per_sm(PerDevice& setup, K kernel, int smem, int* bp) {
  return setup.run(
      [&](int& b) {
        if (smem > 48 * 1024) {
          const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
          if (e != cudaSuccess) return e;
        }
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kThreads, smem) != cudaSuccess || b < 1)
          b = 1;
        cudaGetLastError();
        return cudaSuccess;
      },
      bp);
}

// 2-D TMA map over the bf16 tensor x [rows, cols]: 128x128 boxes, no swizzle,
// zero fill past the edges.  False if unavailable (cols % 8 != 0 included).
bool make_x_map(CUtensorMap* m, const void* x, int64_t rows, int64_t cols) {
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tma_encoder());
  if (!enc || cols % 8 != 0 || rows >= (int64_t{1} << 31) || cols >= (int64_t{1} << 31)) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
  cuuint32_t box[2] = {kTile, kTile};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FMT, bool CURRENT>
cudaError_t launch_cast_transpose(const void* x, int64_t rows, int64_t cols, void* out, void* out_t,
                                  TensorState* st, uint32_t* err, int num_sms, cudaStream_t s, uint32_t extra_tx) {
  const int64_t tiles = ((rows + kTile - 1) / kTile) * ((cols + kTile - 1) / kTile);
  CUtensorMap map;
  if (make_x_map(&map, x, rows, cols)) {
    static PerDevice setup_t;
    int bp = 1;
    const cudaError_t e = blocks_per_sm(setup_t, amax_cast_transpose_tma<FMT, CURRENT>, kTSmem, &bp);
    if (e != cudaSuccess) return e;
    int64_t grid = tiles;
    if (grid > (int64_t)num_sms * bp) grid = (int64_t)num_sms * bp;
    const cudaError_t le = launch_pdl(amax_cast_transpose_tma<FMT, CURRENT>, dim3((unsigned)grid), dim3(kThreads),
                                      kTSmem, s, map, static_cast<uint8_t*>(out), static_cast<uint8_t*>(out_t),
                                      rows, cols, st, err, extra_tx);
    if (le != cudaSuccess) return le;
  } else {
    static PerDevice setup_r;
    int bp = 1;
    const cudaError_t e = blocks_per_sm(setup_r, amax_cast_transpose<FMT, CURRENT>, 0, &bp);
    if (e != cudaSuccess) return e;
    int64_t grid = tiles;
    if (grid > (int64_t)num_sms * bp) grid = (int64_t)num_sms * bp;
    const cudaError_t le = launch_pdl(amax_cast_transpose<FMT, CURRENT>, dim3((unsigned)grid), dim3(kThreads), 0,
                                      s, static_cast<const uint16_t*>(x), static_cast<uint8_t*>(out),
                                      static_cast<uint8_t*>(out_t), rows, cols, st);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

template <int FMT, bool CURRENT>
cudaError_t launch_cast_t(const RecipeDev& rd, int id, const void* x, int64_t rows, int64_t cols,
                          bool update_now, void* out, void* out_t, int num_sms, cudaStream_t s,
                          uint32_t extra_tx) {
  TensorState* st = rd.states + id;
  float* h = rd.history + (int64_t)id * rd.H;
  const int64_t n = rows * cols;
  // one-pass grid of the flat kernels: one block per kFlatBlockVecs vectors
  const int64_t flat_grid = std::max<int64_t>(1, ((n >> 3) + kFlatBlockVecs - 1) / kFlatBlockVecs);
  if (flat_grid >= (int64_t{1} << 31)) return cudaErrorInvalidValue;
  if (CURRENT) {
    const cudaError_t le =
        launch_pdl(amax_only, dim3((unsigned)flat_grid), dim3(kThreads), 0, s, static_cast<const uint4*>(x), n, st);
    if (le != cudaSuccess) return le;
  }
  if (out_t == nullptr) {
    const cudaError_t le = launch_pdl(amax_cast_flat<FMT, CURRENT>, dim3((unsigned)flat_grid), dim3(kThreads), 0, s,
                                      static_cast<const uint16_t*>(x), static_cast<uint8_t*>(out), n, st);
    if (le != cudaSuccess) return le;
  } else {
    const cudaError_t e = launch_cast_transpose<FMT, CURRENT>(x, rows, cols, out, out_t, st, rd.error, num_sms, s,
                                                              extra_tx);
    if (e != cudaSuccess) return e;
  }
  // update_now: this tensor's history update, stream-ordered after every block
  if (update_now) {
    const cudaError_t le = launch_pdl(update_scales_kernel, dim3(1), dim3(32), 0, s, st, h, 1, rd.H, rd.algo);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_amax_cast(const RecipeDev& rd, int tensor_id, const void* x, int64_t rows,
                             int64_t cols, int dtype, bool current, bool update_now, void* out,
                             void* out_t, int num_sms, cudaStream_t s, uint32_t extra_tx) {
  if (dtype == kE4M3) {
    return current ? launch_cast_t<kE4M3, true>(rd, tensor_id, x, rows, cols, update_now, out, out_t, num_sms, s,
                                                extra_tx)
                   : launch_cast_t<kE4M3, false>(rd, tensor_id, x, rows, cols, update_now, out, out_t, num_sms, s,
                                                 extra_tx);
  }
  return current ? launch_cast_t<kE5M2, true>(rd, tensor_id, x, rows, cols, update_now, out, out_t, num_sms, s,
                                              extra_tx)
                 : launch_cast_t<kE5M2, false>(rd, tensor_id, x, rows, cols, update_now, out, out_t, num_sms, s,
                                               extra_tx);
}

cudaError_t launch_update_scales(const RecipeDev& rd, cudaStream_t s) {
  const int threads = 128;
  const int grid = (rd.num_tensors + threads - 1) / threads;
  const cudaError_t le =
      launch_pdl(update_scales_kernel, dim3(grid), dim3(threads), 0, s, rd.states, rd.history, rd.num_tensors, rd.H,
                 rd.algo);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}

cudaError_t launch_set_state(const RecipeDev& rd, int tensor_id, const float* history_dev,
                             float scale, int dtype, cudaStream_t s) {
  set_state_kernel<<<1, 32, 0, s>>>(rd.states + tensor_id, rd.history + (int64_t)tensor_id * rd.H,
                                    history_dev, rd.H, scale, dtype);
  return cudaGetLastError();
}

}  // namespace fp8lin
