// mx_kernels.cu -- MX block scaling: quantisation and the block-scaled GEMM.
//
// "FP8 and low-precision formats" (aiunderstanding.org), format overview:
// frameworks scale values into the FP8 window with per-tensor *or per-block*
// factors, and the MX formats (MXFP8 among them) share one scale per small
// block of elements.  The page gives no rule for the block scale; this library
// reads it as the per-tensor rule of "4.2 Hopper I -- Transformer Engine / FP8"
// (S4.2.4: scale = FP8_MAX / amax) restricted to powers of two:
//   block  = 32 consecutive elements of a row (the row's last block may be
//            shorter, down to 16 elements);
//   k      = the largest integer in [-127, 127] with amax_block * 2^k <= FP8_MAX
//            (-127 when there is none: an Inf or NaN in the block);
//   scale  = one E8M0 byte 127 - k, the block's dequantisation factor 2^-k;
//   q      = round_to_fp8(x * 2^k), saturating RNE (the product is exact).
// Because 2^k never exceeds FP8_MAX / amax, no element of a finite block
// saturates.
//
// Scale layout ("atoms"): the scales of a [rows, cols] matrix form
// ceil(rows/128) x ceil(cols/128) atoms of 512 bytes, atom-row-major; atom
// (i, j) covers rows 128i..128i+127 and blocks 4j..4j+3, and the scale of row r,
// block b lies at byte (r % 32) * 16 + ((r / 32) % 4) * 4 + (b % 4) of its atom.
// That is the order in which tcgen05.cp ... 32x128b.warpx4 spreads one 512-byte
// piece over TMEM for the block-scaled MMA: TMEM lane l (of every lane quarter),
// column c + g holds the four block scales of row 32g + (l % 32).
//
// mx_quantize_kernel: persistent CTAs (three per SM) over 128x128 tiles, with a
// two-buffer TMA ring: while one bf16 tile is quantised the next one's copy is
// in flight.  Per tile, pass 1 takes each row block's and each column block's
// max |x| (bf16 bit patterns, NaN above Inf); the scales are written as two
// atoms (rows of x, rows of x^T); pass 2 writes the codes of x row by row and
// the codes of x^T sixteen rows at a time.
//
// mx_gemm_kernel: the one-CTA tcgen05 GEMM of gemm_tcgen05.cu with block scales:
// per 128-byte K stage the producer also copies one A scale atom and two B
// scale atoms into shared memory (cp.async.bulk, counted on the stage's
// barrier); a copier warp moves them into the stage's TMEM slot with
// tcgen05.cp and signals the MMA warp, which issues
// tcgen05.mma.kind::mxf8f6f4.block_scale.scale_vec::1X (M=128, N=256, K=32),
// choosing the byte of the scale word by the scale-factor IDs of the
// instruction descriptor.  The 128x256 fp32 partial sum takes 256 TMEM
// columns and the scale slots 48 more, so only ONE partial buffer fits in the
// 512 columns: at each promotion (every kMxGroup k-blocks) the MMA warp waits
// for the sixteen epilogue warps to read the partial into registers, which they
// do with four 16-column TMEM loads each before they release it.  One lane
// polls the partial's barrier and wakes the others through a named barrier.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "state.cuh"
#include "tc_ptx.cuh"

namespace fp8lin {
namespace {

// ------------------------------------------------------------ shared math --
// Block exponent k from the bf16 bit pattern of max|x| (sign cleared):
// amax = (1 + f/128) * 2^(e-127) for a normal pattern, and FP8_MAX =
// 1.75 * 2^emax, so amax * 2^k <= FP8_MAX  <=>  k <= emax + 127 - e when
// f <= 96 (1 + f/128 <= 1.75), one less otherwise.  A zero or subnormal amax
// fits at k = 127; an Inf/NaN pattern fits nowhere (-127).
__device__ __forceinline__ int mx_exponent(uint32_t abs_bits, int emax) {
  // abs_bits <= 0x7FFF; a zero or subnormal pattern (e = 0) gives k >= 127
  const int e = static_cast<int>(abs_bits >> 7);
  const int k = min(emax + 127 - e - ((abs_bits & 0x7Fu) > 96u ? 1 : 0), 127);
  return e == 255 ? -127 : k;
}
// 2^k as bf16 bits, k in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ uint16_t pow2bf(int k) {
  return static_cast<uint16_t>(k >= -126 ? (k + 127) << 7 : 0x0040);
}
// The two bf16 values of w times the bf16 power of two s, as fp32: a
// mixed-precision multiply-add with a -0 addend (which keeps the sign of a
// zero product).  A bf16 x bf16 product fits fp32's significand, so the result
// is exact except below fp32's normal range, where every FP8 code is 0 anyway.
// It replaces unpacking each value to fp32 with integer instructions.
__device__ __forceinline__ void mul2_bf16(uint32_t w, uint16_t s, float& lo, float& hi) {
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "fma.rn.f32.bf16 %0, l, %3, 0f80000000;\n\t"
      "fma.rn.f32.bf16 %1, h, %3, 0f80000000;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(w), "h"(s));
}
// One bf16 value (the low half of w if HI is false, else the high half) times
// the bf16 power of two s, as mul2_bf16 computes it.
template <bool HI>
__device__ __forceinline__ float mul1_bf16(uint32_t w, uint16_t s) {
  float r;
  if (HI)
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %1;\n\t"
        "fma.rn.f32.bf16 %0, h, %2, 0f80000000;\n\t}"
        : "=f"(r)
        : "r"(w), "h"(s));
  else
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %1;\n\t"
        "fma.rn.f32.bf16 %0, l, %2, 0f80000000;\n\t}"
        : "=f"(r)
        : "r"(w), "h"(s));
  return r;
}
// Byte offset of (row r, block b) inside its 512-byte scale atom.
__device__ __forceinline__ int atom_offset(int r, int b) {
  return (r & 31) * 16 + ((r >> 5) & 3) * 4 + (b & 3);
}

// ------------------------------------------------------------ quantiser ----
constexpr int kQTile = 128;
constexpr int kQThreads = 256;    // 8 warps, 16 rows of a tile each
#ifndef FP8LIN_MXQ_BUFS
#define FP8LIN_MXQ_BUFS 2
#endif
#ifndef FP8LIN_MXQ_CTAS
#define FP8LIN_MXQ_CTAS 3
#endif
constexpr int kQBufs = FP8LIN_MXQ_BUFS;       // bf16 tiles in flight per CTA
constexpr int kQCtasPerSm = FP8LIN_MXQ_CTAS;
constexpr int kQTileBytes = kQTile * kQTile * 2;
constexpr int kQSmem = kQBufs * kQTileBytes + 128;  // + alignment slack

// Scratch of one tile's scale computation (static shared memory).
struct QScratch {
  alignas(16) uint8_t atom_q[512];
  alignas(16) uint8_t atom_t[512];
  uint16_t rowmax[kQTile][4];  // max |x| bits of row r's block b
  uint16_t colmax[8][kQTile];  // per warp: max |x| bits of a column over its 16 rows
  uint16_t rowmul[kQTile][4];  // 2^k of row block (r, b), bf16 bits
  uint16_t colmul[4][kQTile];  // 2^k of column block (j, c), bf16 bits
};

// Quantise one 128 x 128 tile held in shared memory (bf16 bits, row-major).
// Warp w owns tile rows 16w..16w+15 (inside column block w/2), lane l columns
// 4l..4l+3 (inside row block l/8); the warp's values stay in registers from the
// maxima pass to the code pass.  Once they are, the tile's buffer is reused to
// stage the x^T codes so that each x^T row leaves as one 128-byte line: word
// (c, u) (rows 4u..4u+3 of column c) sits at word c*32 + (u ^ (c / 4 % 32)),
// which keeps both the column-wise writes and the row-wise reads free of bank
// conflicts.
template <int FMT, bool TRANS>
__device__ __forceinline__ void mx_quantize_tile(uint16_t* __restrict__ tile, QScratch& sc, int rows,
                                                 int cols, int tile_r, int tile_c, uint8_t* __restrict__ q,
                                                 uint8_t* __restrict__ q_scale, uint8_t* __restrict__ qt,
                                                 uint8_t* __restrict__ qt_scale) {
  constexpr int emax = FMT == kE4M3 ? 8 : 15;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int atoms_c = (cols + kQTile - 1) / kQTile;
  const int atoms_r = (rows + kQTile - 1) / kQTile;
  const int col0 = tile_c * kQTile;
  const int row0 = tile_r * kQTile;

  // ---- pass 1: maxima of row blocks (8-lane groups) and column partials ------
  uint2 d[16];
  uint32_t cm01 = 0u, cm23 = 0u;  // column maxima, two 16-bit halves each
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    // two rows at a time: their maxima share one word through the 8-lane reduction
    const int r = 16 * warp + i;
    d[i] = *reinterpret_cast<const uint2*>(tile + r * kQTile + 4 * lane);
    d[i + 1] = *reinterpret_cast<const uint2*>(tile + (r + 1) * kQTile + 4 * lane);
    const uint32_t a01 = d[i].x & 0x7FFF7FFFu, a23 = d[i].y & 0x7FFF7FFFu;
    const uint32_t b01 = d[i + 1].x & 0x7FFF7FFFu, b23 = d[i + 1].y & 0x7FFF7FFFu;
    cm01 = __vmaxu2(cm01, __vmaxu2(a01, b01));
    cm23 = __vmaxu2(cm23, __vmaxu2(a23, b23));
    const uint32_t ma = __vmaxu2(a01, a23), mb = __vmaxu2(b01, b23);
    // low half: row r, high half: row r + 1
    uint32_t m = __vmaxu2(__byte_perm(ma, mb, 0x5410), __byte_perm(ma, mb, 0x7632));
    m = __vmaxu2(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = __vmaxu2(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    m = __vmaxu2(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
    if ((lane & 7) == 0) {
      sc.rowmax[r][lane >> 3] = static_cast<uint16_t>(m & 0xFFFFu);
      sc.rowmax[r + 1][lane >> 3] = static_cast<uint16_t>(m >> 16);
    }
  }
  if (TRANS) {
    *reinterpret_cast<uint2*>(&sc.colmax[warp][4 * lane]) = make_uint2(cm01, cm23);
  }
  __syncthreads();

  // ---- block exponents: 512 row blocks (and 512 column blocks), 2 (4) per thread
#pragma unroll
  for (int p = threadIdx.x; p < 4 * kQTile; p += kQThreads) {
    const int r = p >> 2, b = p & 3;
    const int k = mx_exponent(sc.rowmax[r][b], emax);
    sc.rowmul[r][b] = pow2bf(k);
    sc.atom_q[atom_offset(r, b)] = static_cast<uint8_t>(127 - k);
  }
  if (TRANS) {
#pragma unroll
    for (int p = threadIdx.x; p < 4 * kQTile; p += kQThreads) {
      const int j = p >> 7, c = p & (kQTile - 1);
      const uint32_t m =
          max(static_cast<uint32_t>(sc.colmax[2 * j][c]), static_cast<uint32_t>(sc.colmax[2 * j + 1][c]));
      const int k = mx_exponent(m, emax);
      sc.colmul[j][c] = pow2bf(k);
      sc.atom_t[atom_offset(c, j)] = static_cast<uint8_t>(127 - k);
    }
  }
  __syncthreads();

  // ---- scales: one atom of x, one of x^T -------------------------------------
  if (warp == 0) {
    const uint4 v = reinterpret_cast<const uint4*>(sc.atom_q)[lane];
    reinterpret_cast<uint4*>(q_scale + (static_cast<int64_t>(tile_r) * atoms_c + tile_c) * 512)[lane] = v;
  } else if (TRANS && warp == 1) {
    const uint4 v = reinterpret_cast<const uint4*>(sc.atom_t)[lane];
    reinterpret_cast<uint4*>(qt_scale + (static_cast<int64_t>(tile_c) * atoms_r + tile_r) * 512)[lane] = v;
  }

  // ---- pass 2: codes from the registers --------------------------------------
  const int c = col0 + 4 * lane;
  const bool col_ok = c < cols;  // cols % 16 == 0: four columns in or out together
  uint16_t cmul[4] = {0, 0, 0, 0};
  if (TRANS) {
    const uint2 v = *reinterpret_cast<const uint2*>(&sc.colmul[warp >> 1][4 * lane]);
    cmul[0] = static_cast<uint16_t>(v.x & 0xFFFFu);
    cmul[1] = static_cast<uint16_t>(v.x >> 16);
    cmul[2] = static_cast<uint16_t>(v.y & 0xFFFFu);
    cmul[3] = static_cast<uint16_t>(v.y >> 16);
  }
  uint32_t tq[4][4];  // x^T codes: column t, rows 4g..4g+3 of the warp's sixteen
#pragma unroll
  for (int g = 0; g < 4; ++g) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint2 v = d[4 * g + i];
      const int r = 16 * warp + 4 * g + i;
      const uint16_t mr = sc.rowmul[r][lane >> 3];
      if (col_ok && row0 + r < rows) {
        float p0, p1, p2, p3;
        mul2_bf16(v.x, mr, p0, p1);
        mul2_bf16(v.y, mr, p2, p3);
        const uint32_t w = __byte_perm(cvt_fp8x2<FMT>(p0, p1), cvt_fp8x2<FMT>(p2, p3), 0x5410);
        __stcs(reinterpret_cast<unsigned int*>(q + static_cast<int64_t>(row0 + r) * cols + c), w);
      }
    }
    if (TRANS) {
      // column t's values of rows 4g..4g+3
      float y[4][4];  // [t][i]
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint2 u = d[4 * g + i];
        y[0][i] = mul1_bf16<false>(u.x, cmul[0]);
        y[1][i] = mul1_bf16<true>(u.x, cmul[1]);
        y[2][i] = mul1_bf16<false>(u.y, cmul[2]);
        y[3][i] = mul1_bf16<true>(u.y, cmul[3]);
      }
#pragma unroll
      for (int t = 0; t < 4; ++t)
        tq[t][g] = __byte_perm(cvt_fp8x2<FMT>(y[t][0], y[t][1]), cvt_fp8x2<FMT>(y[t][2], y[t][3]), 0x5410);
    }
  }
  if (TRANS) {
    uint32_t* stage = reinterpret_cast<uint32_t*>(tile);  // every warp has its values in registers
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int g = 0; g < 4; ++g) stage[(4 * lane + t) * 32 + ((4 * warp + g) ^ lane)] = tq[t][g];
    __syncthreads();
    // x^T row c of the tile (rows row0..row0+127 of x): 32 words, one per lane
    const int rows_here = min(kQTile, rows - row0);  // a multiple of 16
#pragma unroll 4
    for (int i = 0; i < kQTile / 8; ++i) {
      const int cc = warp * (kQTile / 8) + i;
      if (col0 + cc < cols && 4 * lane < rows_here)
        __stcs(reinterpret_cast<unsigned int*>(qt + static_cast<int64_t>(col0 + cc) * rows + row0 + 4 * lane),
               stage[cc * 32 + (lane ^ ((cc >> 2) & 31))]);
    }
  }
}

// Persistent over tiles t = blockIdx.x, + gridDim.x, ...: while a tile is
// quantised the next one's TMA copy is in flight in the other buffer.
template <int FMT, bool TRANS>
__global__ void __launch_bounds__(kQThreads, kQCtasPerSm) mx_quantize_kernel(
    const __grid_constant__ CUtensorMap tmX, int rows, int cols, uint8_t* __restrict__ q,
    uint8_t* __restrict__ q_scale, uint8_t* __restrict__ qt, uint8_t* __restrict__ qt_scale,
    uint32_t* err) {
  extern __shared__ uint8_t qsmem_raw[];
  uint16_t* tiles = reinterpret_cast<uint16_t*>(qsmem_raw + ((128u - (smem_u32(qsmem_raw) & 127u)) & 127u));
  __shared__ QScratch sc;
  __shared__ alignas(8) uint64_t bar[kQBufs];
  __shared__ int give_up;

  const int atoms_c = (cols + kQTile - 1) / kQTile;
  const int num_tiles = atoms_c * ((rows + kQTile - 1) / kQTile);
  if (threadIdx.x == 0) {
    for (int b = 0; b < kQBufs; ++b) mbar_init(&bar[b], 1);
    fence_mbar_init();
    give_up = 0;
    for (int b = 0; b < kQBufs; ++b) {
      const int t = blockIdx.x + b * gridDim.x;
      if (t < num_tiles) {
        mbar_expect_tx(&bar[b], kQTileBytes);
        tma_load_2d(tiles + b * kQTile * kQTile, &tmX, &bar[b], (t % atoms_c) * kQTile, (t / atoms_c) * kQTile);
      }
    }
  }
  __syncthreads();
  int it = 0;
  for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
    const int b = it % kQBufs;
    const uint32_t parity = static_cast<uint32_t>(it / kQBufs) & 1u;
    if (threadIdx.x == 0) {
      const uint32_t addr = smem_u32(&bar[b]);
      const uint64_t t0 = gtimer();
      bool ok = mbar_try_wait(addr, parity);
      while (!ok && gtimer() - t0 < kTimeoutNs) ok = mbar_try_wait(addr, parity);
      if (!ok) {
        // record the time-out; wait (bounded) for this CTA's copies in flight
        atomicOr(err, kErrTimeoutMx);
        for (int i = 0; i < kQBufs; ++i) {
          const int tt = t + i * gridDim.x;
          if (tt >= num_tiles) break;
          const uint32_t a2 = smem_u32(&bar[(it + i) % kQBufs]);
          const uint32_t p2 = static_cast<uint32_t>((it + i) / kQBufs) & 1u;
          const uint64_t t1 = gtimer();
          while (!mbar_try_wait(a2, p2) && gtimer() - t1 < kTimeoutNs) {
          }
        }
        give_up = 1;
      }
    }
    __syncthreads();
    if (give_up) return;
    mx_quantize_tile<FMT, TRANS>(tiles + b * kQTile * kQTile, sc, rows, cols, t / atoms_c, t % atoms_c, q,
                                 q_scale, qt, qt_scale);
    if (TRANS) fence_async_smem();  // staging stores before the next TMA write of this buffer
    __syncthreads();                // the tile buffer and the scratch are free again
    if (threadIdx.x == 0) {
      const int tn = t + kQBufs * gridDim.x;
      if (tn < num_tiles) {
        mbar_expect_tx(&bar[b], kQTileBytes);
        tma_load_2d(tiles + b * kQTile * kQTile, &tmX, &bar[b], (tn % atoms_c) * kQTile, (tn / atoms_c) * kQTile);
      }
    }
  }
}

// ------------------------------------------------------------ MX GEMM ------
constexpr int kMxBM = 128;
constexpr int kMxBN = 256;
constexpr int kMxBK = 128;  // bytes = elements = four MMAs of K = 32
#ifndef FP8LIN_MX_STAGES
#define FP8LIN_MX_STAGES 4
#endif
#ifndef FP8LIN_MX_STORE_ROWS
#define FP8LIN_MX_STORE_ROWS 8
#endif
#ifndef FP8LIN_MX_EPI_SLEEP
#define FP8LIN_MX_EPI_SLEEP 0
#endif
#ifndef FP8LIN_MX_EPI_WAIT
#define FP8LIN_MX_EPI_WAIT 1
#endif
constexpr int kMxStages = FP8LIN_MX_STAGES;
constexpr int kMxABytes = kMxBM * kMxBK;
constexpr int kMxBBytes = kMxBN * kMxBK;
constexpr int kMxStageBytes = kMxABytes + kMxBBytes;
constexpr int kMxSfBytes = 512 + 1024;  // one A atom, two B atoms per stage
constexpr int kMxEpiWarps = 16;         // four per TMEM lane quarter, 64 columns each
// warps: producer, MMA issuer, sixteen epilogue warps, scale copier
constexpr int kMxCopierWarp = 2 + kMxEpiWarps;
constexpr int kMxThreads = (kMxCopierWarp + 1) * 32;
constexpr int kMxEpiCols = kMxBN / 4;
constexpr int kMxStoreRows = FP8LIN_MX_STORE_ROWS;  // output rows per TMA store
constexpr int kMxStaging = kMxStoreRows * 128;      // per epilogue warp: rows x 128 bytes
constexpr int kMxEpiSleepNs = FP8LIN_MX_EPI_SLEEP;  // back-off of the partial wait (0: none)
// How the epilogue waits for a finished partial: 0 every warp polls, 1 one
// lane polls and releases the sixteen warps through a named barrier (measured
// 10 % faster on 8192x4096x16384: sixteen polling warps slow the MMA warp).
constexpr int kMxEpiWait = FP8LIN_MX_EPI_WAIT;
static_assert(32 % kMxStoreRows == 0 && kMxStoreRows % 8 == 0, "store rows: 8, 16 or 32");
#ifndef FP8LIN_MX_KGROUP
#define FP8LIN_MX_KGROUP 16
#endif
constexpr int kMxGroup = FP8LIN_MX_KGROUP;  // k-blocks per TMEM partial
constexpr int kMxGroupM = 16;               // 128-row tiles per raster group
constexpr int kMxTmemCols = 512;
constexpr int kMxSfCol0 = kMxBN;            // scale slots after the partial-sum columns
constexpr int kMxBarBytes = 192;
constexpr int kMxSmem = kMxStages * kMxStageBytes + kMxEpiWarps * kMxStaging + kMxStages * kMxSfBytes +
                        kMxBarBytes + 1024;
static_assert(kMxSmem <= 232448, "shared memory per block exceeded");
static_assert(kMxSfCol0 + 16 * kMxStages <= kMxTmemCols, "TMEM columns exceeded");
static_assert((3 * kMxStages + 3) * 8 + 12 <= kMxBarBytes, "barrier area too small");

// Shared-memory descriptor of one 512-byte scale atom: 32 rows of 16 bytes,
// no swizzle, 8-row core matrices 128 bytes apart (both offsets 128 bytes).
__device__ __forceinline__ uint64_t sdesc_atom(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128 >> 4) << 16;
  d |= static_cast<uint64_t>(128 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version (sm_100 family); swizzle none
  return d;
}
// Copy one 32 x 128-bit piece of shared memory into TMEM columns
// [taddr, taddr + 4) of every lane quarter.
__device__ __forceinline__ void tmem_copy_atom(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}\n" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Bounded wait with a short sleeping back-off.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                unsigned ns) {
  const uint32_t addr = smem_u32(bar);
  const uint64_t t0 = gtimer();
  for (;;) {
    if (mbar_try_wait(addr, parity)) return true;
    __nanosleep(ns);
    if (*abort_flag) return false;
    if (gtimer() - t0 > kTimeoutNs) return false;
  }
}

__device__ __forceinline__ void mx_tile_coords(int t, int tiles_m, int tiles_n, int& mb, int& nb) {
  const int group = kMxGroupM * tiles_n;
  const int g = t / group;
  const int first_m = g * kMxGroupM;
  const int gm = min(kMxGroupM, tiles_m - first_m);
  const int r = t - g * group;
  mb = first_m + r % gm;
  nb = r / gm;
}

// Store this warp's 32 rows x 64 columns (row0 + lane, from colw): TMA stores of
// kMxStoreRows-row x 128-byte blocks staged in the warp's buffer (128-byte
// swizzle), or, when the output layout does not allow TMA, direct per-row
// stores.
template <bool F32>
__device__ __forceinline__ void mx_store(const float (&acc)[kMxEpiCols], uint8_t* buf, const CUtensorMap* tmD,
                                         int tma_store, void* D, int64_t ldd, int row0, int colw, int lane,
                                         int M, int N) {
  if (tma_store) {
    constexpr int CPB = F32 ? 32 : 64;  // columns per 128-byte block
    constexpr int VPC = CPB / 8;        // values per 16-byte chunk
    const uint32_t sbase = smem_u32(buf);
#pragma unroll
    for (int b = 0; b < kMxEpiCols / CPB; ++b) {
      const int cb = colw + b * CPB;
      if (cb >= N) break;  // warp-uniform
#pragma unroll
      for (int c = 0; c < 32 / kMxStoreRows; ++c) {
        if (lane == 0) bulk_wait_read_all();  // the previous block has left the buffer
        __syncwarp();
        if (lane / kMxStoreRows == c) {
          const int rr = lane % kMxStoreRows;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float* a = acc + b * CPB + j * VPC;
            uint32_t w[4];
            if (F32) {
#pragma unroll
              for (int t = 0; t < 4; ++t) w[t] = __float_as_uint(a[t]);
            } else {
#pragma unroll
              for (int t = 0; t < 4; ++t) w[t] = bf16x2_bits(a[2 * t], a[2 * t + 1]);
            }
            st_shared_v4(sbase + rr * 128 + ((j ^ (rr & 7)) << 4), w[0], w[1], w[2], w[3]);
          }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) tma_store_2d(tmD, sbase, cb, row0 + c * kMxStoreRows);
      }
    }
    return;
  }
  const int row = row0 + lane;
  if (row >= M) return;
  for (int c = 0; c < kMxEpiCols; ++c) {
    const int col = colw + c;
    if (col >= N) break;
    if (F32)
      static_cast<float*>(D)[static_cast<int64_t>(row) * ldd + col] = acc[c];
    else
      static_cast<__nv_bfloat16*>(D)[static_cast<int64_t>(row) * ldd + col] = __float2bfloat16_rn(acc[c]);
  }
}

template <bool F32>
__global__ void __launch_bounds__(kMxThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const uint8_t* __restrict__ a_scale,
                   const uint8_t* __restrict__ b_scale, void* __restrict__ D, int64_t ldd, int M, int N, int K,
                   int tiles_m, int tiles_n, uint32_t idesc, uint32_t* err, int tma_store) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* staging = smem + kMxStages * kMxStageBytes;    // 1024-aligned
  uint8_t* sf = staging + kMxEpiWarps * kMxStaging;       // per stage: A atom, B atom 0, B atom 1
  uint64_t* full = reinterpret_cast<uint64_t*>(sf + kMxStages * kMxSfBytes);
  uint64_t* empty = full + kMxStages;
  uint64_t* tfull = empty + kMxStages;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint64_t* sfready = drain + 1;  // per stage: its data landed and its scales are in TMEM
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sfready + kMxStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_flag = abort_flag + 1;  // the leader's wait result (kMxEpiWait == 1)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = tiles_m * tiles_n;
  const int nk = (K + kMxBK - 1) / kMxBK;
  const int atoms_k = nk;                        // scale atoms per 128 rows
  const int atoms_n = (N + 127) / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kMxEpiWarps);
    mbar_init(drain, 1);
    for (int s = 0; s < kMxStages; ++s) mbar_init(&sfready[s], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // finite scales in the B slots a ragged last tile does not load (those rows
  // are zero-filled and their products discarded)
  for (int i = threadIdx.x; i < kMxStages * kMxSfBytes / 4; i += kMxThreads)
    reinterpret_cast<uint32_t*>(sf)[i] = 0u;
  fence_async_smem();
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kMxTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        int mb, nb;
        mx_tile_coords(t, tiles_m, tiles_n, mb, nb);
        const bool b_hi = 2 * nb + 1 < atoms_n;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&full[stage], kMxStageBytes + (b_hi ? kMxSfBytes : 1024));
          uint8_t* sA = smem + stage * kMxStageBytes;
          uint8_t* sS = sf + stage * kMxSfBytes;
          tma_load_2d(sA, &tmA, &full[stage], kb * kMxBK, mb * kMxBM);
          tma_load_2d(sA + kMxABytes, &tmB, &full[stage], kb * kMxBK, nb * kMxBN);
          bulk_load(sS, a_scale + (static_cast<int64_t>(mb) * atoms_k + kb) * 512, 512, &full[stage]);
          bulk_load(sS + 512, b_scale + (static_cast<int64_t>(2 * nb) * atoms_k + kb) * 512, 512, &full[stage]);
          if (b_hi)
            bulk_load(sS + 1024, b_scale + (static_cast<int64_t>(2 * nb + 1) * atoms_k + kb) * 512, 512,
                      &full[stage]);
          ++issued;
          if (++stage == kMxStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(err, kErrTimeoutMx);
        const int pending = issued < kMxStages ? (int)issued : kMxStages;
        for (int i = 1; i <= pending; ++i) {
          int s = stage - i;
          uint32_t ph = phase;
          if (s < 0) {
            s += kMxStages;
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
      int grp = 0;
      bool ok = true;
      bool issued_any = false;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        for (int kb = 0; kb < nk; ++kb) {
          const int kg = kb % kMxGroup;
          if (kg == 0) {  // the epilogue has read the previous partial
            if (!mbar_wait(tempty, (grp & 1) ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          // the copier completes this after the stage's data landed and its
          // scales reached TMEM
          if (!mbar_wait(&sfready[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * kMxStageBytes);
          const uint64_t adesc = sdesc_sw128(a_addr);
          const uint64_t bdesc = sdesc_sw128(a_addr + kMxABytes);
          const uint32_t sfa = tmem_base + static_cast<uint32_t>(kMxSfCol0 + 16 * stage);
          const uint32_t sfb = sfa + 4u;
#pragma unroll
          for (int k = 0; k < kMxBK / 32; ++k) {
            // byte k of each scale word belongs to the k-th 32-element block
            const uint32_t id = idesc | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
            mma_mx(tmem_base, adesc + 2u * k, bdesc + 2u * k, id, sfa, sfb, (kg | k) ? 1u : 0u);
          }
          issued_any = true;
          mma_commit(&empty[stage]);
          if (++stage == kMxStages) {
            stage = 0;
            phase ^= 1u;
          }
          if (kg == kMxGroup - 1 || kb == nk - 1) {
            mma_commit(tfull);  // partial complete
            ++grp;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(err, kErrTimeoutMx);
        if (issued_any) {
          mma_commit(drain);
          const uint32_t addr = smem_u32(drain);
          const uint64_t t0 = gtimer();
          while (!mbar_try_wait(addr, 0) && gtimer() - t0 < kTimeoutNs) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == kMxCopierWarp) {
    // -------------------------------------------------------- scale copier --
    // Moves each stage's block scales from shared memory into the stage's TMEM
    // slot, off the MMA thread (a copy issued there right before the stage's
    // MMAs stalled the tensor pipe: 0.43 ms against 0.36 ms on 8192x4096x16384).
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      long copied = 0;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        for (int kb = 0; kb < nk; ++kb) {
          // the stage's data has landed, so the MMAs of its previous use (which
          // read this TMEM slot) completed before the producer refilled it
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t s_addr = smem_u32(sf + stage * kMxSfBytes);
          const uint32_t slot = tmem_base + static_cast<uint32_t>(kMxSfCol0 + 16 * stage);
          tmem_copy_atom(slot, sdesc_atom(s_addr));              // A rows 0..127
          tmem_copy_atom(slot + 4u, sdesc_atom(s_addr + 512));   // B rows 0..127
          tmem_copy_atom(slot + 8u, sdesc_atom(s_addr + 1024));  // B rows 128..255
          mma_commit(&sfready[stage]);
          ++copied;
          if (++stage == kMxStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(err, kErrTimeoutMx);
        if (copied > 0) {  // the last copies complete before TMEM is freed
          int s0 = stage - 1;
          uint32_t p0 = phase;
          if (s0 < 0) {
            s0 += kMxStages;
            p0 ^= 1u;
          }
          const uint32_t addr = smem_u32(&sfready[s0]);
          const uint64_t t0 = gtimer();
          while (!mbar_try_wait(addr, p0) && gtimer() - t0 < kTimeoutNs) {
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue --
    const int quarter = warp & 3;                // TMEM lanes this warp may read
    const int cg = (warp - 2) >> 2;              // which 64 of the 256 columns
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                           static_cast<uint32_t>(cg * kMxEpiCols);
    const int ngroups = (nk + kMxGroup - 1) / kMxGroup;
    int grp = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
      int mb, nb;
      mx_tile_coords(t, tiles_m, tiles_n, mb, nb);
      float acc[kMxEpiCols];
#pragma unroll
      for (int j = 0; j < kMxEpiCols; ++j) acc[j] = 0.0f;
      for (int g = 0; g < ngroups; ++g, ++grp) {
        int w = 1;
        if (kMxEpiWait == 1) {
          // one lane polls; the others sleep in the named barrier
          if (warp == 2 && lane == 0)
            *epi_flag = (kMxEpiSleepNs > 0 ? mbar_wait_sleep(tfull, grp & 1, abort_flag, kMxEpiSleepNs)
                                           : mbar_wait(tfull, grp & 1, abort_flag))
                            ? 1
                            : 0;
          named_bar_sync(1, kMxEpiWarps * 32);
          w = *epi_flag;
        } else {
          if (lane == 0)
            w = (kMxEpiSleepNs > 0 ? mbar_wait_sleep(tfull, grp & 1, abort_flag, kMxEpiSleepNs)
                                   : mbar_wait(tfull, grp & 1, abort_flag))
                    ? 1
                    : 0;
          w = __shfl_sync(0xFFFFFFFFu, w, 0);
        }
        if (!w) {
          if (lane == 0) {
            *abort_flag = 1;
            atomicOr(err, kErrTimeoutMx);
          }
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < kMxEpiCols / 16; ++h) {
          uint32_t r[16];
          tmem_ld16(taddr + static_cast<uint32_t>(16 * h), r);
          tmem_ld_wait();
          if (h == kMxEpiCols / 16 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty);  // the MMAs may overwrite the partial now
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[16 * h + j] = __fadd_rn(acc[16 * h + j], __uint_as_float(r[j]));
        }
      }
      if (!ok) break;
      mx_store<F32>(acc, staging + (warp - 2) * kMxStaging, &tmD, tma_store, D, ldd, mb * kMxBM + quarter * 32,
                    nb * kMxBN + cg * kMxEpiCols, lane, M, N);
      __syncwarp();
    }
    if (tma_store && lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kMxTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Pair kernel: a cluster of two CTAs (the two SMs of a TPC) computes a 256x256
// output tile with tcgen05.mma.cta_group::2 ... .block_scale (M=256, N=256,
// K=32), in 256-byte K stages: eight MMAs per stage wait and commit once (the
// per-tensor pair kernel measured 20-30 % from that).  CTA r loads A rows
// [128r, 128r+128) and B rows [128r, 128r+128) of the tile, and the block
// scales of its A rows and of all 256 of the tile's B rows (each CTA's MMA
// reads the scales of every column it computes from its own TMEM), all by TMA
// counted on the leader's stage barrier.
// The leader's copier warp moves a stage's scales into both CTAs' TMEM with
// tcgen05.cp.cta_group::2 (the same shared-memory offset of each CTA to the
// same TMEM column of each); the leader's MMA warp issues the MMAs.  TMEM holds
// one 128x256 fp32 partial per CTA (256 columns) and three stages of scale
// slots, so the partial is single-buffered as in the one-CTA kernel: at each
// promotion (every 2048 of K) the MMA warp waits until the sixteen epilogue
// warps of both CTAs have read it.
// ---------------------------------------------------------------------------
constexpr int kMx2BK = 256;                            // K bytes per stage: eight MMAs of K = 32
constexpr int kMx2Stages = 3;
constexpr int kMx2Half = 128 * kMx2BK;                 // A or B half per CTA per stage
constexpr int kMx2SfA = 1024;                          // two atoms: this CTA's 128 rows x 8 blocks
constexpr int kMx2SfB = 2048;                          // four atoms: the tile's 256 B rows x 8 blocks
constexpr int kMx2StageBytes = 2 * kMx2Half + kMx2SfA + kMx2SfB;
constexpr int kMx2StageAlloc = (kMx2StageBytes + 1023) / 1024 * 1024;  // stages stay 1024-aligned
constexpr int kMx2Group = 2048 / kMx2BK;               // stages per TMEM partial (K = 2048)
constexpr int kMx2SlotCols = 24;                       // TMEM columns of one stage's scales
constexpr int kMx2Smem = kMx2Stages * kMx2StageAlloc + kMxEpiWarps * kMxStaging + kMxBarBytes + 1024;
static_assert(kMx2Smem <= 232448, "shared memory per block exceeded");
static_assert(kMxSfCol0 + kMx2SlotCols * kMx2Stages <= kMxTmemCols, "TMEM columns exceeded");
static_assert((3 * kMx2Stages + 3) * 8 + 12 <= kMxBarBytes, "barrier area too small");

__device__ __forceinline__ void tmem_copy_atom2(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void mma_mx_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}\n" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mx_tile_coords2(int t, int tiles_m, int tiles_n, int& mb, int& nb) {
  constexpr int G = 8;  // 256-row tiles per raster group
  const int group = G * tiles_n;
  const int g = t / group;
  const int first_m = g * G;
  const int gm = min(G, tiles_m - first_m);
  const int r = t - g * group;
  mb = first_m + r % gm;
  nb = r / gm;
}

template <bool F32>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kMxThreads, 1)
    mx_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                        const __grid_constant__ CUtensorMap tmD, void* __restrict__ D, int64_t ldd, int M, int N,
                        int K, int tiles_m, int tiles_n, uint32_t idesc, uint32_t* err, int tma_store) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* staging = smem + kMx2Stages * kMx2StageAlloc;  // 1024-aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + kMxEpiWarps * kMxStaging);
  uint64_t* empty = full + kMx2Stages;
  uint64_t* tfull = empty + kMx2Stages;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint64_t* sfready = drain + 1;  // per stage: its scales are in both CTAs' TMEM
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sfready + kMx2Stages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0 = leader
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;
  const int num_tiles = tiles_m * tiles_n;
  const int nk = (K + kMx2BK - 1) / kMx2BK;
  const int atoms_k = (K + 127) / 128;  // scale atoms per 128 rows

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMx2Stages; ++s) {
      mbar_init(&full[s], 1);     // leader: one arrive.expect_tx, both CTAs' bytes
      mbar_init(&empty[s], 1);    // one multicast commit per use
      mbar_init(&sfready[s], 1);  // leader: the copier's commit
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 2 * kMxEpiWarps);  // leader: epilogue warps of both CTAs
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmSA);
    prefetch_tmap(&tmSB);
  }
  if (warp == 1) {
    tmem_alloc2(tmem_slot, kMxTmemCols);
    tmem_relinquish2();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers exist before anyone signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long issued = 0;
      bool ok = true;
      for (int t = cluster; ok && t < num_tiles; t += nclusters) {
        int mb, nb;
        mx_tile_coords2(t, tiles_m, tiles_n, mb, nb);
        const int m0 = mb * 256 + 128 * static_cast<int>(rank), n0 = nb * 256 + 128 * static_cast<int>(rank);
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t leader_full = mapa_shared(smem_u32(&full[stage]), 0);
          if (rank == 0) mbar_expect_tx(&full[stage], 2 * kMx2StageBytes);
          uint8_t* sA = smem + stage * kMx2StageAlloc;
          uint8_t* sS = sA + 2 * kMx2Half;
          const int k0 = kb * kMx2BK;  // boxes past K read zeros
          for (int h = 0; h < 2; ++h) {
            tma_load_2d_pair(sA + h * (128 * 128), &tmA, leader_full, k0 + 128 * h, m0);
            tma_load_2d_pair(sA + kMx2Half + h * (128 * 128), &tmB, leader_full, k0 + 128 * h, n0);
          }
          // scale atoms (2kb, 2kb+1) of a 128-row block rb: rows 2 (rb atoms_k + 2kb) .. +3
          // of the scale array viewed as 256-byte rows
          const int ka = 2 * kb;
          tma_load_2d_pair(sS, &tmSA, leader_full, 0, 2 * ((2 * mb + static_cast<int>(rank)) * atoms_k + ka));
          for (int hh = 0; hh < 2; ++hh)
            tma_load_2d_pair(sS + kMx2SfA + 1024 * hh, &tmSB, leader_full, 0, 2 * ((2 * nb + hh) * atoms_k + ka));
          ++issued;
          if (++stage == kMx2Stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(err, kErrTimeoutMx);
      }
      if (!ok && rank == 0) {
        // the leader's stage barriers count both CTAs' copies: let them land
        const int pending = issued < kMx2Stages ? (int)issued : kMx2Stages;
        for (int i = 1; i <= pending; ++i) {
          int s = stage - i;
          uint32_t ph = phase;
          if (s < 0) {
            s += kMx2Stages;
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
      for (int t = cluster; ok && t < num_tiles; t += nclusters) {
        for (int kb = 0; kb < nk; ++kb) {
          const int kg = kb % kMx2Group;
          if (kg == 0) {  // both CTAs' epilogues have read the previous partial
            if (!mbar_wait_cl(tempty, (grp & 1) ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          if (!mbar_wait(&sfready[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * kMx2StageAlloc);
          const uint32_t b_addr = a_addr + kMx2Half;
          const uint32_t slot = tmem_base + static_cast<uint32_t>(kMxSfCol0 + kMx2SlotCols * stage);
#pragma unroll
          for (int k = 0; k < kMx2BK / 32; ++k) {
            // K = 32 further on: 32 bytes inside a box's swizzled rows (the next
            // box every four steps); block k's scale is byte k % 4 of atom k / 4
            const uint64_t ad = sdesc_sw128(a_addr + (k >> 2) * (128 * 128)) + 2u * (k & 3);
            const uint64_t bd = sdesc_sw128(b_addr + (k >> 2) * (128 * 128)) + 2u * (k & 3);
            const uint32_t id = idesc | (static_cast<uint32_t>(k & 3) << 4) | (static_cast<uint32_t>(k & 3) << 29);
            const uint32_t sfa = slot + 4u * (k >> 2);
            const uint32_t sfb = slot + 8u + 8u * (k >> 2);  // B rows 0-127, then 128-255
            mma_mx_pair(tmem_base, ad, bd, id, sfa, sfb, (kg | k) ? 1u : 0u);
          }
          issued_any = true;
          mma_commit_pair(&empty[stage], 0x3);
          if (++stage == kMx2Stages) {
            stage = 0;
            phase ^= 1u;
          }
          if (kg == kMx2Group - 1 || kb == nk - 1) {
            mma_commit_pair(tfull, 0x3);  // partial complete, in both CTAs
            ++grp;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(err, kErrTimeoutMx);
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
  } else if (warp == kMxCopierWarp) {
    // ------------------------------------------- scale copier (leader only) --
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      long copied = 0;
      for (int t = cluster; ok && t < num_tiles; t += nclusters) {
        for (int kb = 0; kb < nk; ++kb) {
          // both CTAs' data landed, so the MMAs of the stage's previous use
          // (which read these TMEM slots) completed before it was refilled
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t s_addr = smem_u32(smem + stage * kMx2StageAlloc + 2 * kMx2Half);
          const uint32_t slot = tmem_base + static_cast<uint32_t>(kMxSfCol0 + kMx2SlotCols * stage);
          tmem_copy_atom2(slot, sdesc_atom(s_addr));              // A, blocks 0-3 of the stage
          tmem_copy_atom2(slot + 4u, sdesc_atom(s_addr + 512));   // A, blocks 4-7
          // per four blocks: B rows 0-127 then rows 128-255 of the tile
          tmem_copy_atom2(slot + 8u, sdesc_atom(s_addr + kMx2SfA));
          tmem_copy_atom2(slot + 12u, sdesc_atom(s_addr + kMx2SfA + 1024));
          tmem_copy_atom2(slot + 16u, sdesc_atom(s_addr + kMx2SfA + 512));
          tmem_copy_atom2(slot + 20u, sdesc_atom(s_addr + kMx2SfA + 1536));
          mma_commit_pair(&sfready[stage], 0x1);
          ++copied;
          if (++stage == kMx2Stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(err, kErrTimeoutMx);
        if (copied > 0) {  // the last copies complete before TMEM is freed
          int s0 = stage - 1;
          uint32_t p0 = phase;
          if (s0 < 0) {
            s0 += kMx2Stages;
            p0 ^= 1u;
          }
          const uint32_t addr = smem_u32(&sfready[s0]);
          const uint64_t t0 = gtimer();
          while (!mbar_try_wait(addr, p0) && gtimer() - t0 < kTimeoutNs) {
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue --
    const int quarter = warp & 3;    // TMEM lanes this warp may read
    const int cg = (warp - 2) >> 2;  // which 64 of the 256 columns
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                           static_cast<uint32_t>(cg * kMxEpiCols);
    const int ngroups = (nk + kMx2Group - 1) / kMx2Group;
    const uint32_t leader_tempty = mapa_shared(smem_u32(tempty), 0);
    int grp = 0;
    bool ok = true;
    for (int t = cluster; ok && t < num_tiles; t += nclusters) {
      int mb, nb;
      mx_tile_coords2(t, tiles_m, tiles_n, mb, nb);
      float acc[kMxEpiCols];
#pragma unroll
      for (int j = 0; j < kMxEpiCols; ++j) acc[j] = 0.0f;
      for (int g = 0; g < ngroups; ++g, ++grp) {
        // one lane polls; the others sleep in the named barrier
        if (warp == 2 && lane == 0) *epi_flag = mbar_wait_cl(tfull, grp & 1, abort_flag) ? 1 : 0;
        named_bar_sync(1, kMxEpiWarps * 32);
        const int w = *epi_flag;
        named_bar_sync(2, kMxEpiWarps * 32);  // everyone has read the flag before it is rewritten
        if (!w) {
          if (lane == 0) {
            *abort_flag = 1;
            atomicOr(err, kErrTimeoutMx);
          }
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < kMxEpiCols / 16; ++h) {
          uint32_t r[16];
          tmem_ld16(taddr + static_cast<uint32_t>(16 * h), r);
          tmem_ld_wait();
          if (h == kMxEpiCols / 16 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(leader_tempty);  // the MMAs may overwrite the partial now
          }
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            float& lo = acc[16 * h + j];
            float& hi = acc[16 * h + j + 1];
            f2_unpack(f2_add(f2_pack(lo, hi), f2_pack(__uint_as_float(r[j]), __uint_as_float(r[j + 1]))), lo, hi);
          }
        }
      }
      if (!ok) break;
      mx_store<F32>(acc, staging + (warp - 2) * kMxStaging, &tmD, tma_store, D, ldd,
                    mb * 256 + 128 * static_cast<int>(rank) + quarter * 32, nb * 256 + cg * kMxEpiCols, lane, M, N);
      __syncwarp();
    }
    if (tma_store && lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync_all();  // no signal may target a CTA that has left
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc2(tmem_base, kMxTmemCols);
  }
}

// ------------------------------------------------------------ host side ----
// 128 x 128 bf16 tiles of a [rows, cols] matrix, no swizzle, zeros outside.
bool make_bf16_tile_map(CUtensorMap* m, const void* x, int64_t rows, int64_t cols) {
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tma_encoder());
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
  cuuint32_t box[2] = {kQTile, kQTile};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FMT, bool TRANS>
cudaError_t launch_q(const CUtensorMap& m, int grid, int rows, int cols, void* q, void* q_scale, void* q_t,
                     void* q_t_scale, uint32_t* err, cudaStream_t s) {
  static PerDevice setup;
  const cudaError_t attr_err = setup.run([](int&) {
    return cudaFuncSetAttribute(mx_quantize_kernel<FMT, TRANS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kQSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  mx_quantize_kernel<FMT, TRANS><<<grid, kQThreads, kQSmem, s>>>(
      m, rows, cols, static_cast<uint8_t*>(q), static_cast<uint8_t*>(q_scale), static_cast<uint8_t*>(q_t),
      static_cast<uint8_t*>(q_t_scale), err);
  return cudaGetLastError();
}

// The scale array of an MX matrix viewed as rows of 256 bytes (two rows per
// 512-byte atom); boxes of four rows = the two atoms of one 128-row block that
// a 256-byte K stage needs.  No swizzle; rows past the end read zeros.
bool make_scale_map(CUtensorMap* m, const void* sc, int64_t bytes) {
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tma_encoder());
  if (!enc) return false;
  cuuint64_t dims[2] = {256, static_cast<cuuint64_t>(bytes / 256)};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {256, 4};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(sc), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The two-CTA kernel runs only when FP8LIN_MX_KERNEL=pair (and M > 128).
// Measured at 8192 x 4096 x 16384 in one call, it ran 2847-2859 TFLOP/s
// against the one-CTA kernel's 2960-2966: both hold a single TMEM partial, so
// the MMAs stop at every promotion until the epilogue has read it, and the
// pair adds a cluster-wide round trip to that stop.
bool mx_pair_allowed() {
  static const bool v = [] {
    const char* e = getenv("FP8LIN_MX_KERNEL");
    return e != nullptr && strcmp(e, "pair") == 0;
  }();
  return v;
}

template <bool F32>
cudaError_t launch_mx_gemm_pair(const MxGemmArgs& g, int num_sms, cudaStream_t s, const char** detail) {
  static PerDevice setup;
  int resident = 0;
  const cudaError_t attr_err = setup.run(
      [&](int& r) {
        const cudaError_t e =
            cudaFuncSetAttribute(mx_gemm_pair_kernel<F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMx2Smem);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t c = {};
        c.blockDim = dim3(kMxThreads);
        c.gridDim = dim3(2);
        c.dynamicSmemBytes = kMx2Smem;
        c.stream = s;
        if (cudaOccupancyMaxActiveClusters(&r, mx_gemm_pair_kernel<F32>, &c) != cudaSuccess) r = 0;
        cudaGetLastError();
        return cudaSuccess;
      },
      &resident);
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap ma, mb, msa, msb, md;
  const int64_t atoms_k = (g.K + 127) / 128;
  if (!make_map(&ma, g.A, g.K, g.M, g.lda, 128, 128) || !make_map(&mb, g.B, g.K, g.N, g.ldb, 128, 128) ||
      !make_scale_map(&msa, g.a_scale, ((g.M + 127) / 128) * atoms_k * 512) ||
      !make_scale_map(&msb, g.b_scale, ((g.N + 127) / 128) * atoms_k * 512)) {
    if (detail) *detail = "cuTensorMapEncodeTiled failed (driver entry point or arguments)";
    return cudaErrorInvalidValue;
  }
  memset(&md, 0, sizeof md);
  const int tma_store = make_out_map(&md, g.D, g.M, g.N, g.ldd, F32 ? 4 : 2, kMxStoreRows) ? 1 : 0;
  const int tiles_m = static_cast<int>((g.M + 255) / 256);
  const int tiles_n = static_cast<int>((g.N + 255) / 256);
  const int tiles = tiles_m * tiles_n;
  // block-scaled instruction descriptor: A/B formats at bits 7 and 10, K-major
  // A and B, N >> 3 at bit 17, UE8M0 scales (bit 23), M >> 4 at bit 24 (M =
  // 256 across the pair); the scale-factor IDs (bits 4 and 29) are set per MMA
  const uint32_t idesc = (static_cast<uint32_t>(g.a_dtype) << 7) | (static_cast<uint32_t>(g.b_dtype) << 10) |
                         (static_cast<uint32_t>(256 >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(256 >> 4) << 24);
  const int cap = resident > 0 && resident < num_sms / 2 ? resident : num_sms / 2;
  const int clusters = tiles < cap ? tiles : cap;
  mx_gemm_pair_kernel<F32><<<2 * clusters, kMxThreads, kMx2Smem, s>>>(
      ma, mb, msa, msb, md, g.D, g.ldd, static_cast<int>(g.M), static_cast<int>(g.N), static_cast<int>(g.K),
      tiles_m, tiles_n, idesc, g.error, tma_store);
  return cudaGetLastError();
}

template <bool F32>
cudaError_t launch_mx_gemm_t(const MxGemmArgs& g, int num_sms, cudaStream_t s, const char** detail) {
  if (g.M > kMxBM && num_sms >= 2 && mx_pair_allowed()) return launch_mx_gemm_pair<F32>(g, num_sms, s, detail);
  static PerDevice setup;
  const cudaError_t attr_err = setup.run([](int&) {
    return cudaFuncSetAttribute(mx_gemm_kernel<F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMxSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap ma, mb, md;
  if (!make_map(&ma, g.A, g.K, g.M, g.lda, kMxBK, kMxBM) || !make_map(&mb, g.B, g.K, g.N, g.ldb, kMxBK, kMxBN)) {
    if (detail) *detail = "cuTensorMapEncodeTiled failed (driver entry point or arguments)";
    return cudaErrorInvalidValue;
  }
  memset(&md, 0, sizeof md);
  const int tma_store = make_out_map(&md, g.D, g.M, g.N, g.ldd, F32 ? 4 : 2, kMxStoreRows) ? 1 : 0;
  const int tiles_m = static_cast<int>((g.M + kMxBM - 1) / kMxBM);
  const int tiles_n = static_cast<int>((g.N + kMxBN - 1) / kMxBN);
  const int tiles = tiles_m * tiles_n;
  // block-scaled instruction descriptor: A/B formats at bits 7 and 10, K-major
  // A and B, N >> 3 at bit 17, UE8M0 scales (bit 23), M >> 4 at bit 24; the
  // scale-factor IDs (bits 4 and 29) are set per MMA
  const uint32_t idesc = (static_cast<uint32_t>(g.a_dtype) << 7) | (static_cast<uint32_t>(g.b_dtype) << 10) |
                         (static_cast<uint32_t>(kMxBN >> 3) << 17) | (1u << 23) |
                         (static_cast<uint32_t>(kMxBM >> 4) << 24);
  const int grid = tiles < num_sms ? tiles : num_sms;
  mx_gemm_kernel<F32><<<grid, kMxThreads, kMxSmem, s>>>(
      ma, mb, md, static_cast<const uint8_t*>(g.a_scale), static_cast<const uint8_t*>(g.b_scale), g.D, g.ldd,
      static_cast<int>(g.M), static_cast<int>(g.N), static_cast<int>(g.K), tiles_m, tiles_n, idesc, g.error,
      tma_store);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mx_quantize(const void* x, int64_t rows, int64_t cols, int dtype, void* q, void* q_scale,
                               void* q_t, void* q_t_scale, uint32_t* error, int num_sms, cudaStream_t s,
                               const char** detail) {
  CUtensorMap m;
  if (!make_bf16_tile_map(&m, x, rows, cols)) {
    if (detail) *detail = "cuTensorMapEncodeTiled failed (driver entry point or arguments)";
    return cudaErrorInvalidValue;
  }
  const int64_t tiles = ((cols + kQTile - 1) / kQTile) * ((rows + kQTile - 1) / kQTile);
  const int grid = static_cast<int>(tiles < static_cast<int64_t>(num_sms) * kQCtasPerSm ? tiles
                                                                                      : num_sms * kQCtasPerSm);
  const int r = static_cast<int>(rows), c = static_cast<int>(cols);
  const bool tr = q_t != nullptr;
  if (dtype == kE4M3)
    return tr ? launch_q<kE4M3, true>(m, grid, r, c, q, q_scale, q_t, q_t_scale, error, s)
              : launch_q<kE4M3, false>(m, grid, r, c, q, q_scale, q_t, q_t_scale, error, s);
  return tr ? launch_q<kE5M2, true>(m, grid, r, c, q, q_scale, q_t, q_t_scale, error, s)
            : launch_q<kE5M2, false>(m, grid, r, c, q, q_scale, q_t, q_t_scale, error, s);
}

cudaError_t launch_mx_gemm(const MxGemmArgs& g, int num_sms, cudaStream_t s, const char** detail) {
  return g.d_kind == 1 ? launch_mx_gemm_t<true>(g, num_sms, s, detail)
                       : launch_mx_gemm_t<false>(g, num_sms, s, detail);
}

}  // namespace fp8lin
