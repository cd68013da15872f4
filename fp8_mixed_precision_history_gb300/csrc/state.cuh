// state.cuh -- device-resident scaling state of one recipe, and the launch
// entry points the C ABI layer calls.  Internal to libfp8lin.
#pragma once

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <cuda_runtime.h>
#include <mutex>
#include <utility>

namespace fp8lin {

constexpr int kE4M3 = 0;
constexpr int kE5M2 = 1;
constexpr float kMaxE4M3 = 448.0f;    // largest finite OCP E4M3 value (0x7E)
constexpr float kMaxE5M2 = 57344.0f;  // largest finite OCP E5M2 value (0x7B)

// Device error word bits (recipe-wide).
constexpr uint32_t kErrTimeoutGemm = 1u;
constexpr uint32_t kErrTimeoutCast = 2u;
constexpr uint32_t kErrTimeoutMx = 4u;

// One tensor's scaling state.  Amax values are stored as fp32 bit patterns of
// non-negative numbers so that unsigned max == float max (NaN above +Inf).
struct alignas(128) TensorState {
  // Read by every thread of a cast or a GEMM (one 32-byte sector).
  float scale;           // scale of the next delayed cast
  float scale_inv;       // 1/scale (fp32 RN)
  float cast_scale;      // scale of the most recent cast
  float cast_scale_inv;  // its reciprocal (GEMM dequant factor)
  uint32_t amax_last;    // amax pushed by the most recent update
  int32_t dtype;
  int32_t recorded;
  int32_t head;          // ring index of the newest history entry
  // Current scaling's first pass: (epoch + 1) << 32 | amax bits, by atomicMax.
  // A new pass's tag exceeds every older value, so the word is never reset.
  // The cast pass reads it through the read-only path (it is final by then).
  unsigned long long amax_acc;
  uint32_t epoch;        // current-scaling casts completed on this tensor
  uint32_t pad0_[5];
  // Folded into by the blocks of every cast (atomics): kept off the sectors
  // above, so that the reads there do not queue behind them.
  uint32_t amax_pending; // max amax recorded since the last history update
  uint32_t pad1_;
  unsigned long long n_sat;    // counts since the last update
  unsigned long long n_und;
  unsigned long long n_sat_last;
  unsigned long long n_und_last;
};
static_assert(sizeof(TensorState) == 128, "one 128-byte line per tensor");

struct RecipeDev {
  TensorState* states;  // [num_tensors]
  float* history;       // [num_tensors][H] ring buffers
  uint32_t* error;      // device error word
  int num_tensors;
  int H;
  int algo;             // 0 = max, 1 = most recent
};

// Set-up that each device needs once (a kernel's shared-memory opt-in is a
// per-device function attribute; occupancy is a per-device query).  run(fn)
// calls fn(value) the first time it runs with a given device current and
// returns fn's status, and the int fn stored, on that call and every later one.
constexpr int kMaxDevices = 64;
struct PerDevice {
  std::once_flag once[kMaxDevices];
  cudaError_t err[kMaxDevices] = {};
  int value[kMaxDevices] = {};
  template <typename F>
  cudaError_t run(F fn, int* value_out = nullptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [&] { err[dev] = fn(value[dev]); });
    if (value_out != nullptr) *value_out = value[dev];
    return err[dev];
  }
};

// ---- launchers (cast_kernels.cu) -------------------------------------------
// extra_tx: 0, or the bytes by which the TMA cast-transpose over-states its
// first stage (the test hook of fp8_debug_inject_stall).
cudaError_t launch_amax_cast(const RecipeDev& rd, int tensor_id, const void* x, int64_t rows,
                             int64_t cols, int dtype, bool current, bool update_now, void* out,
                             void* out_t, int num_sms, cudaStream_t s, uint32_t extra_tx);
cudaError_t launch_update_scales(const RecipeDev& rd, cudaStream_t s);
cudaError_t launch_set_state(const RecipeDev& rd, int tensor_id, const float* history_dev,
                             float scale, int dtype, cudaStream_t s);

// ---- launcher (gemm_tcgen05.cu) --------------------------------------------
struct GemmArgs {
  const void* A; int a_dtype; int64_t lda;
  const void* B; int b_dtype; int64_t ldb;
  bool a_mn, b_mn;  // false: A [M, K] / B [N, K] (K contiguous); true: A [K, M] / B [K, N]
  int64_t M, N, K;
  void* D; int d_kind; int64_t ldd;  // d_kind: 0 bf16, 1 fp32, 2 E4M3 codes, 3 E5M2 codes
  const TensorState* sa; const TensorState* sb;
  TensorState* s_out;  // nullptr: no fused amax; FP8 outputs: the output tensor
  uint32_t* error;
  uint32_t extra_tx;   // 0, or the fp8_debug_inject_stall over-statement of the first stage
  int act;             // 0 none, 1 GELU (aux: bf16 pre-activation out), 2 GELU' (aux: bf16 in)
  void* aux;           // bf16 [M, N], row stride ld_aux elements; nullptr when unused
  int64_t ld_aux;
  // Split tail (two-CTA kernel): the recipe's workspace of sk_slots partial
  // tiles (kSplitSlotBytes each), their flags (kSplitSlotFlags each), and two
  // more words after the flags: the launch epoch the flags compare against
  // and the exit count that advances it (see the kernel).
  float* sk_ws;
  uint32_t* sk_flags;
  int sk_slots;
};
// One split-tail slot: a 256 x 256 fp32 partial tile, and one flag per
// epilogue warp of the CTA pair.
constexpr size_t kSplitSlotBytes = size_t{256} * 256 * 4;
constexpr int kSplitSlotFlags = 16;
// Returns cudaSuccess or an error; a failure to encode a TMA descriptor is
// reported as cudaErrorInvalidValue with *detail set.
cudaError_t launch_gemm(const GemmArgs& g, int num_sms, cudaStream_t s, const char** detail);

// ---- launchers (mx_kernels.cu): MX block scaling -----------------------------
// Quantise a bf16 [rows, cols] matrix with one power-of-two scale per 32
// elements of a row, and optionally its transpose with its own scales.
cudaError_t launch_mx_quantize(const void* x, int64_t rows, int64_t cols, int dtype, void* q,
                               void* q_scale, void* q_t, void* q_t_scale, uint32_t* error, int num_sms,
                               cudaStream_t s, const char** detail);
struct MxGemmArgs {
  const void* A; int a_dtype; int64_t lda; const void* a_scale;
  const void* B; int b_dtype; int64_t ldb; const void* b_scale;
  int64_t M, N, K;
  void* D; int d_kind; int64_t ldd;  // d_kind: 0 bf16, 1 fp32
  uint32_t* error;
};
cudaError_t launch_mx_gemm(const MxGemmArgs& g, int num_sms, cudaStream_t s, const char** detail);

// ---- launchers (grad_allreduce.cu): FP8 gradient all-reduce steps ----------
cudaError_t launch_grad_amax(const void* g, int64_t n, float* amax, int num_sms, cudaStream_t s);
cudaError_t launch_grad_quantize(const void* g, int64_t n, const float* amax, int world, void* codes,
                                 int64_t padded_n, float* scale, int num_sms, cudaStream_t s);
cudaError_t launch_grad_reduce(const void* recv, int world, int64_t chunk, void* out, int num_sms,
                               cudaStream_t s);
cudaError_t launch_grad_dequantize(const void* codes, int64_t n, const float* scale, int world, int average,
                                   void* out, int num_sms, cudaStream_t s);

// The driver's cuTensorMapEncodeTiled (PFN_cuTensorMapEncodeTiled_v12000),
// looked up once through the runtime; nullptr if unavailable.
void* tma_encoder();

// Record the calling thread's error detail (read by fp8_last_error_message).
void set_last_error(const char* msg);

// Launch with programmatic dependent launch allowed: the kernel may begin
// while the previous kernel on the stream is finishing, and waits for it
// (griddepcontrol.wait) before it touches memory; so a launch's latency and a
// GEMM's set-up (barriers, TMEM, tensor maps) overlap the previous kernel's
// tail.  Every kernel launched this way waits before its first global access.
// FP8LIN_PDL=0 launches plainly.
inline bool pdl_enabled() {
  static const bool v = [] {
    const char* e = getenv("FP8LIN_PDL");
    return !(e != nullptr && strcmp(e, "0") == 0);
  }();
  return v;
}
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (pdl_enabled()) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace fp8lin
