// fp8lin_api.cu -- the C ABI (include/fp8lin.h): argument checks, recipe state
// ownership, and kernel launches.  No arithmetic of the method happens here;
// every step of the path runs in the kernels of cast_kernels.cu,
// gemm_tcgen05.cu, mx_kernels.cu and grad_allreduce.cu.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "fp8lin.h"
#include "state.cuh"

using fp8lin::RecipeDev;
using fp8lin::TensorState;

struct fp8_recipe {
  RecipeDev dev;
  int format;
  int num_sms;
  int device;
  float* dev_hist_in;       // H floats: staging for fp8_set_state
  TensorState* host_state;  // pinned staging for fp8_get_state
  float* host_hist;         // pinned, H floats
  uint32_t* host_err;       // pinned
  uint32_t stall_once;      // fp8_debug_inject_stall: bit 0 next TMA cast-transpose, bit 1 next GEMM
  // the GEMM's split-tail workspace: one partial tile and its flags per CTA
  // pair of the device, then the launch epoch and exit count
  float* sk_ws;
  uint32_t* sk_flags;
  int sk_slots;
};

namespace {

thread_local std::string g_msg;

fp8_status_t fail(fp8_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_msg = buf;
  return st;
}

fp8_status_t cuda_fail(cudaError_t e, const char* where) {
  return fail(FP8_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaStream_t as_stream(fp8_stream_t s) { return static_cast<cudaStream_t>(s); }

fp8_status_t check_id(const fp8_recipe_t* r, int32_t id, const char* what) {
  if (id < 0 || id >= r->dev.num_tensors)
    return fail(FP8_ERR_INVALID, "%s %d out of range [0, %d)", what, id, r->dev.num_tensors);
  return FP8_OK;
}

bool valid_dtype(int32_t d) { return d == FP8_E4M3 || d == FP8_E5M2; }

// Read (and clear) the recipe's device error word; the stream is synchronised.
fp8_status_t read_device_error(fp8_recipe_t* r, cudaStream_t s) {
  cudaError_t e = cudaMemcpyAsync(r->host_err, r->dev.error, sizeof(uint32_t),
                                  cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e, "reading device error word");
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  const uint32_t w = *r->host_err;
  if (w != 0u) {
    cudaMemsetAsync(r->dev.error, 0, sizeof(uint32_t), s);
    cudaStreamSynchronize(s);
    return fail(FP8_ERR_TIMEOUT, "device wait exceeded its limit (error bits 0x%x: %s%s%s)", w,
                (w & fp8lin::kErrTimeoutGemm) ? "gemm " : "", (w & fp8lin::kErrTimeoutCast) ? "cast " : "",
                (w & fp8lin::kErrTimeoutMx) ? "mx" : "");
  }
  return FP8_OK;
}

}  // namespace

void fp8lin::set_last_error(const char* msg) { g_msg = msg ? msg : ""; }

extern "C" {

const char* fp8_status_string(fp8_status_t st) {
  switch (st) {
    case FP8_OK: return "ok";
    case FP8_ERR_INVALID: return "invalid argument";
    case FP8_ERR_UNSUPPORTED: return "unsupported";
    case FP8_ERR_CUDA: return "CUDA error";
    case FP8_ERR_TIMEOUT: return "device wait timed out";
    case FP8_ERR_NOMEM: return "out of memory";
  }
  return "unknown status";
}

const char* fp8_last_error_message(void) { return g_msg.c_str(); }

fp8_status_t fp8_recipe_create(fp8_recipe_t** out, int32_t format, int32_t amax_history_len,
                               int32_t algo, int32_t num_tensors, fp8_stream_t stream) {
  g_msg.clear();
  if (!out) return fail(FP8_ERR_INVALID, "out is NULL");
  *out = nullptr;
  if (format != FP8_RECIPE_HYBRID && format != FP8_RECIPE_E4M3)
    return fail(FP8_ERR_INVALID, "unknown recipe format %d", format);
  if (algo != FP8_AMAX_MAX && algo != FP8_AMAX_MOST_RECENT)
    return fail(FP8_ERR_INVALID, "unknown amax algorithm %d", algo);
  if (amax_history_len < 1 || amax_history_len > 1024)
    return fail(FP8_ERR_INVALID, "amax_history_len %d not in [1, 1024]", amax_history_len);
  if (num_tensors < 1 || num_tensors > 65536)
    return fail(FP8_ERR_INVALID, "num_tensors %d not in [1, 65536]", num_tensors);
  cudaStream_t s = as_stream(stream);

  fp8_recipe_t* r = static_cast<fp8_recipe_t*>(calloc(1, sizeof(fp8_recipe_t)));
  if (!r) return fail(FP8_ERR_NOMEM, "host allocation");
  r->format = format;
  r->dev.num_tensors = num_tensors;
  r->dev.H = amax_history_len;
  r->dev.algo = algo;
  cudaError_t e = cudaGetDevice(&r->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&r->num_sms, cudaDevAttrMultiProcessorCount, r->device);
  if (e != cudaSuccess) {
    free(r);
    return cuda_fail(e, "querying the device");
  }
  const size_t st_bytes = sizeof(TensorState) * num_tensors;
  const size_t h_bytes = sizeof(float) * static_cast<size_t>(num_tensors) * amax_history_len;
  bool ok = cudaMalloc(&r->dev.states, st_bytes) == cudaSuccess &&
            cudaMalloc(&r->dev.history, h_bytes) == cudaSuccess &&
            cudaMalloc(&r->dev.error, sizeof(uint32_t)) == cudaSuccess &&
            cudaMalloc(&r->dev_hist_in, sizeof(float) * amax_history_len) == cudaSuccess &&
            cudaMallocHost(&r->host_state, sizeof(TensorState)) == cudaSuccess &&
            cudaMallocHost(&r->host_hist, sizeof(float) * amax_history_len) == cudaSuccess &&
            cudaMallocHost(&r->host_err, sizeof(uint32_t)) == cudaSuccess;
  r->sk_slots = r->num_sms / 2 > 0 ? r->num_sms / 2 : 1;
  ok = ok && cudaMalloc(&r->sk_ws, fp8lin::kSplitSlotBytes * r->sk_slots) == cudaSuccess &&
       cudaMalloc(&r->sk_flags, sizeof(uint32_t) * (fp8lin::kSplitSlotFlags * r->sk_slots + 2)) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    fp8_recipe_destroy(r);
    return fail(FP8_ERR_NOMEM, "device or pinned allocation of recipe state failed");
  }
  // initial state: history 0, scales 1, nothing recorded
  TensorState init;
  memset(&init, 0, sizeof init);
  init.scale = init.scale_inv = init.cast_scale = init.cast_scale_inv = 1.0f;
  init.head = amax_history_len - 1;
  init.dtype = FP8_E4M3;
  TensorState* host_init = static_cast<TensorState*>(malloc(st_bytes));
  if (!host_init) {
    fp8_recipe_destroy(r);
    return fail(FP8_ERR_NOMEM, "host allocation");
  }
  for (int i = 0; i < num_tensors; ++i) host_init[i] = init;
  e = cudaMemcpyAsync(r->dev.states, host_init, st_bytes, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(r->dev.history, 0, h_bytes, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(r->dev.error, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(r->sk_flags, 0, sizeof(uint32_t) * (fp8lin::kSplitSlotFlags * r->sk_slots + 2), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  free(host_init);
  if (e != cudaSuccess) {
    fp8_recipe_destroy(r);
    return cuda_fail(e, "initialising recipe state");
  }
  *out = r;
  return FP8_OK;
}

fp8_status_t fp8_recipe_destroy(fp8_recipe_t* r) {
  g_msg.clear();
  if (!r) return FP8_OK;
  cudaError_t e = cudaDeviceSynchronize();
  if (r->dev.states) cudaFree(r->dev.states);
  if (r->dev.history) cudaFree(r->dev.history);
  if (r->dev.error) cudaFree(r->dev.error);
  if (r->dev_hist_in) cudaFree(r->dev_hist_in);
  if (r->host_state) cudaFreeHost(r->host_state);
  if (r->host_hist) cudaFreeHost(r->host_hist);
  if (r->host_err) cudaFreeHost(r->host_err);
  if (r->sk_ws) cudaFree(r->sk_ws);
  if (r->sk_flags) cudaFree(r->sk_flags);
  free(r);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize in destroy");
  return FP8_OK;
}

fp8_status_t fp8_amax_quantize(fp8_recipe_t* r, int32_t tensor_id, const void* x, int64_t rows,
                               int64_t cols, int32_t dtype, int32_t mode, int32_t update_now,
                               void* out, void* out_t, fp8_stream_t stream) {
  g_msg.clear();
  if (!r) return fail(FP8_ERR_INVALID, "recipe is NULL");
  if (fp8_status_t st = check_id(r, tensor_id, "tensor_id")) return st;
  if (!x || !out) return fail(FP8_ERR_INVALID, "x or out is NULL");
  if (!aligned16(x) || !aligned16(out) || (out_t && !aligned16(out_t)))
    return fail(FP8_ERR_INVALID, "x, out and out_t must be 16-byte aligned");
  if (rows < 1 || cols < 1) return fail(FP8_ERR_INVALID, "rows %lld, cols %lld must be >= 1",
                                        (long long)rows, (long long)cols);
  if (rows > (int64_t{1} << 40) / cols) return fail(FP8_ERR_INVALID, "rows*cols too large");
  if (!valid_dtype(dtype)) return fail(FP8_ERR_INVALID, "unknown dtype %d", dtype);
  if (mode != FP8_SCALING_DELAYED && mode != FP8_SCALING_CURRENT)
    return fail(FP8_ERR_INVALID, "unknown scaling mode %d", mode);
  if (r->format == FP8_RECIPE_E4M3 && dtype != FP8_E4M3)
    return fail(FP8_ERR_INVALID, "E4M3 recipe casts every tensor to E4M3");
  uint32_t extra_tx = 0;
  if (out_t != nullptr && cols % 8 == 0 && (r->stall_once & 1u)) {
    r->stall_once &= ~1u;
    extra_tx = 16;
  }
  cudaError_t e = fp8lin::launch_amax_cast(r->dev, tensor_id, x, rows, cols, dtype,
                                           mode == FP8_SCALING_CURRENT, update_now != 0, out,
                                           out_t, r->num_sms, as_stream(stream), extra_tx);
  if (e != cudaSuccess) return cuda_fail(e, "amax/cast launch");
  return FP8_OK;
}

fp8_status_t fp8_gemm_act(fp8_recipe_t* r, int32_t a_id, const void* A, int32_t a_dtype, int32_t a_major,
                          int64_t lda, int32_t b_id, const void* B, int32_t b_dtype, int32_t b_major, int64_t ldb,
                          int64_t M, int64_t N, int64_t K, void* D, int32_t d_dtype, int64_t ldd,
                          int32_t amax_out_id, int32_t act, void* aux, int64_t ld_aux, fp8_stream_t stream) {
  g_msg.clear();
  if (!r) return fail(FP8_ERR_INVALID, "recipe is NULL");
  if (act != FP8_ACT_NONE && act != FP8_ACT_GELU && act != FP8_ACT_DGELU)
    return fail(FP8_ERR_INVALID, "unknown activation %d", act);
  if (act == FP8_ACT_NONE && aux) return fail(FP8_ERR_INVALID, "aux must be NULL without an activation");
  if (act == FP8_ACT_DGELU && !aux)
    return fail(FP8_ERR_INVALID, "FP8_ACT_DGELU needs aux: the forward's bf16 pre-activation");
  if (aux) {
    // the aux tensor moves by TMA in 16-byte pieces: whole pieces per row
    if (!aligned16(aux) || ld_aux < N || ld_aux % 8 != 0 || N % 8 != 0)
      return fail(FP8_ERR_INVALID,
                  "aux must be 16-byte aligned with ld_aux >= N, ld_aux %% 8 == 0 and N %% 8 == 0 "
                  "(N %lld, ld_aux %lld)", (long long)N, (long long)ld_aux);
  }
  if (fp8_status_t st = check_id(r, a_id, "a_id")) return st;
  if (fp8_status_t st = check_id(r, b_id, "b_id")) return st;
  if (amax_out_id != -1)
    if (fp8_status_t st = check_id(r, amax_out_id, "amax_out_id")) return st;
  if (!A || !B || !D) return fail(FP8_ERR_INVALID, "A, B or D is NULL");
  if (!valid_dtype(a_dtype) || !valid_dtype(b_dtype))
    return fail(FP8_ERR_INVALID, "unknown operand dtype (%d, %d)", a_dtype, b_dtype);
  if ((a_major != FP8_K_MAJOR && a_major != FP8_MN_MAJOR) || (b_major != FP8_K_MAJOR && b_major != FP8_MN_MAJOR))
    return fail(FP8_ERR_INVALID, "unknown operand layout (%d, %d)", a_major, b_major);
  if (d_dtype != FP8_OUT_BF16 && d_dtype != FP8_OUT_F32 && d_dtype != FP8_OUT_E4M3 &&
      d_dtype != FP8_OUT_E5M2)
    return fail(FP8_ERR_INVALID, "unknown output dtype %d", d_dtype);
  const bool fp8_out = d_dtype == FP8_OUT_E4M3 || d_dtype == FP8_OUT_E5M2;
  if (fp8_out && amax_out_id < 0)
    return fail(FP8_ERR_INVALID, "an FP8 output needs amax_out_id: the tensor whose scale casts it");
  if (d_dtype == FP8_OUT_E5M2 && r->format == FP8_RECIPE_E4M3)
    return fail(FP8_ERR_INVALID, "E4M3 recipe casts every tensor to E4M3");
  if (M < 1 || N < 1 || M > (1 << 30) || N > (1 << 30))
    return fail(FP8_ERR_INVALID, "M %lld, N %lld must be in [1, 2^30]", (long long)M, (long long)N);
  if (K < 16 || K % 16 != 0 || K > (1 << 30))
    return fail(FP8_ERR_INVALID, "K %lld must be a positive multiple of 16 (<= 2^30)", (long long)K);
  const bool a_mn = a_major == FP8_MN_MAJOR, b_mn = b_major == FP8_MN_MAJOR;
  const int64_t a_row = a_mn ? M : K, b_row = b_mn ? N : K;  // contiguous extent of a stored row
  if (lda < a_row || ldb < b_row || lda % 16 != 0 || ldb % 16 != 0)
    return fail(FP8_ERR_INVALID,
                "lda %lld / ldb %lld must be multiples of 16 and >= the stored row (%lld / %lld)",
                (long long)lda, (long long)ldb, (long long)a_row, (long long)b_row);
  if (!aligned16(A) || !aligned16(B)) return fail(FP8_ERR_INVALID, "A and B must be 16-byte aligned");
  if (ldd < N) return fail(FP8_ERR_INVALID, "ldd %lld < N %lld", (long long)ldd, (long long)N);
  const int esize = d_dtype == FP8_OUT_F32 ? 4 : (fp8_out ? 1 : 2);
  if ((reinterpret_cast<uintptr_t>(D) % esize) != 0) return fail(FP8_ERR_INVALID, "D misaligned");
  const int64_t tiles = ((M + 127) / 128) * ((N + 255) / 256);
  if (tiles > (int64_t{1} << 30)) return fail(FP8_ERR_INVALID, "too many output tiles");

  fp8lin::GemmArgs g;
  g.A = A; g.a_dtype = a_dtype; g.lda = lda;
  g.B = B; g.b_dtype = b_dtype; g.ldb = ldb;
  g.a_mn = a_mn; g.b_mn = b_mn;
  g.M = M; g.N = N; g.K = K;
  g.D = D; g.d_kind = d_dtype; g.ldd = ldd;
  g.sa = r->dev.states + a_id;
  g.sb = r->dev.states + b_id;
  g.s_out = amax_out_id >= 0 ? r->dev.states + amax_out_id : nullptr;
  g.error = r->dev.error;
  g.extra_tx = 0;
  g.act = act;
  g.aux = aux;
  g.ld_aux = ld_aux;
  g.sk_ws = r->sk_ws;
  g.sk_flags = r->sk_flags;
  g.sk_slots = r->sk_slots;
  if (r->stall_once & 2u) {
    r->stall_once &= ~2u;
    g.extra_tx = 16;
  }
  const char* detail = nullptr;
  cudaError_t e = fp8lin::launch_gemm(g, r->num_sms, as_stream(stream), &detail);
  if (e != cudaSuccess) {
    if (detail) return fail(FP8_ERR_CUDA, "gemm: %s", detail);
    return cuda_fail(e, "gemm launch");
  }
  return FP8_OK;
}

fp8_status_t fp8_gemm_layout(fp8_recipe_t* r, int32_t a_id, const void* A, int32_t a_dtype, int32_t a_major,
                             int64_t lda, int32_t b_id, const void* B, int32_t b_dtype, int32_t b_major,
                             int64_t ldb, int64_t M, int64_t N, int64_t K, void* D, int32_t d_dtype,
                             int64_t ldd, int32_t amax_out_id, fp8_stream_t stream) {
  return fp8_gemm_act(r, a_id, A, a_dtype, a_major, lda, b_id, B, b_dtype, b_major, ldb, M, N, K, D, d_dtype,
                      ldd, amax_out_id, FP8_ACT_NONE, nullptr, 0, stream);
}

fp8_status_t fp8_gemm(fp8_recipe_t* r, int32_t a_id, const void* A, int32_t a_dtype, int64_t lda,
                      int32_t b_id, const void* B, int32_t b_dtype, int64_t ldb, int64_t M,
                      int64_t N, int64_t K, void* D, int32_t d_dtype, int64_t ldd,
                      int32_t amax_out_id, fp8_stream_t stream) {
  return fp8_gemm_layout(r, a_id, A, a_dtype, FP8_K_MAJOR, lda, b_id, B, b_dtype, FP8_K_MAJOR, ldb, M, N, K,
                         D, d_dtype, ldd, amax_out_id, stream);
}

int64_t fp8_mx_scale_bytes(int64_t rows, int64_t cols) {
  if (rows < 1 || cols < 1 || rows > (int64_t{1} << 40) / cols) return -1;
  return ((rows + 127) / 128) * ((cols + 127) / 128) * 512;
}

fp8_status_t fp8_mx_quantize(fp8_recipe_t* r, const void* x, int64_t rows, int64_t cols, int32_t dtype,
                             void* q, void* q_scale, void* q_t, void* q_t_scale, fp8_stream_t stream) {
  g_msg.clear();
  if (!r) return fail(FP8_ERR_INVALID, "recipe is NULL");
  if (!x || !q || !q_scale) return fail(FP8_ERR_INVALID, "x, q or q_scale is NULL");
  if ((q_t == nullptr) != (q_t_scale == nullptr))
    return fail(FP8_ERR_INVALID, "q_t and q_t_scale must both be given or both be NULL");
  if (!aligned16(x) || !aligned16(q) || !aligned16(q_scale) || (q_t && (!aligned16(q_t) || !aligned16(q_t_scale))))
    return fail(FP8_ERR_INVALID, "x, q, q_scale, q_t and q_t_scale must be 16-byte aligned");
  if (rows < 1 || cols < 16 || cols % 16 != 0 || cols > (1 << 30) || rows > (1 << 30))
    return fail(FP8_ERR_INVALID, "rows %lld must be in [1, 2^30], cols %lld a multiple of 16 in [16, 2^30]",
                (long long)rows, (long long)cols);
  if (q_t && rows % 16 != 0)
    return fail(FP8_ERR_INVALID, "a transposed copy needs rows %% 16 == 0 (rows %lld)", (long long)rows);
  if (rows > (int64_t{1} << 40) / cols) return fail(FP8_ERR_INVALID, "rows*cols too large");
  if (((rows + 127) / 128) * ((cols + 127) / 128) > (int64_t{1} << 31) - 1)
    return fail(FP8_ERR_INVALID, "too many 128x128 tiles");
  if (!valid_dtype(dtype)) return fail(FP8_ERR_INVALID, "unknown dtype %d", dtype);
  const char* detail = nullptr;
  cudaError_t e = fp8lin::launch_mx_quantize(x, rows, cols, dtype, q, q_scale, q_t, q_t_scale, r->dev.error,
                                             r->num_sms, as_stream(stream), &detail);
  if (e != cudaSuccess) {
    if (detail) return fail(FP8_ERR_CUDA, "mx quantize: %s", detail);
    return cuda_fail(e, "mx quantize launch");
  }
  return FP8_OK;
}

fp8_status_t fp8_mx_gemm(fp8_recipe_t* r, const void* A, int32_t a_dtype, int64_t lda, const void* a_scale,
                         const void* B, int32_t b_dtype, int64_t ldb, const void* b_scale, int64_t M,
                         int64_t N, int64_t K, void* D, int32_t d_dtype, int64_t ldd, fp8_stream_t stream) {
  g_msg.clear();
  if (!r) return fail(FP8_ERR_INVALID, "recipe is NULL");
  if (!A || !B || !D || !a_scale || !b_scale) return fail(FP8_ERR_INVALID, "A, B, D or a scale array is NULL");
  if (!valid_dtype(a_dtype) || !valid_dtype(b_dtype))
    return fail(FP8_ERR_INVALID, "unknown operand dtype (%d, %d)", a_dtype, b_dtype);
  if (d_dtype != FP8_OUT_BF16 && d_dtype != FP8_OUT_F32)
    return fail(FP8_ERR_INVALID, "MX GEMM output dtype %d must be FP8_OUT_BF16 or FP8_OUT_F32", d_dtype);
  if (M < 1 || N < 1 || M > (1 << 30) || N > (1 << 30))
    return fail(FP8_ERR_INVALID, "M %lld, N %lld must be in [1, 2^30]", (long long)M, (long long)N);
  if (K < 16 || K % 16 != 0 || K > (1 << 30))
    return fail(FP8_ERR_INVALID, "K %lld must be a positive multiple of 16 (<= 2^30)", (long long)K);
  if (lda < K || ldb < K || lda % 16 != 0 || ldb % 16 != 0)
    return fail(FP8_ERR_INVALID, "lda %lld / ldb %lld must be >= K and multiples of 16",
                (long long)lda, (long long)ldb);
  if (!aligned16(A) || !aligned16(B) || !aligned16(a_scale) || !aligned16(b_scale))
    return fail(FP8_ERR_INVALID, "A, B and the scale arrays must be 16-byte aligned");
  if (ldd < N) return fail(FP8_ERR_INVALID, "ldd %lld < N %lld", (long long)ldd, (long long)N);
  const int esize = d_dtype == FP8_OUT_F32 ? 4 : 2;
  if ((reinterpret_cast<uintptr_t>(D) % esize) != 0) return fail(FP8_ERR_INVALID, "D misaligned");
  const int64_t tiles = ((M + 127) / 128) * ((N + 255) / 256);
  if (tiles > (int64_t{1} << 30)) return fail(FP8_ERR_INVALID, "too many output tiles");

  fp8lin::MxGemmArgs g;
  g.A = A; g.a_dtype = a_dtype; g.lda = lda; g.a_scale = a_scale;
  g.B = B; g.b_dtype = b_dtype; g.ldb = ldb; g.b_scale = b_scale;
  g.M = M; g.N = N; g.K = K;
  g.D = D; g.d_kind = d_dtype; g.ldd = ldd;
  g.error = r->dev.error;
  const char* detail = nullptr;
  cudaError_t e = fp8lin::launch_mx_gemm(g, r->num_sms, as_stream(stream), &detail);
  if (e != cudaSuccess) {
    if (detail) return fail(FP8_ERR_CUDA, "mx gemm: %s", detail);
    return cuda_fail(e, "mx gemm launch");
  }
  return FP8_OK;
}

// ---- FP8 gradient all-reduce steps (no recipe; the kernels never wait) --------
namespace {
int current_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}
fp8_status_t grad_launch(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return cuda_fail(e, what);
  return FP8_OK;
}
}  // namespace

fp8_status_t fp8_grad_amax(const void* g, int64_t n, float* amax, fp8_stream_t stream) {
  g_msg.clear();
  if (!g || !amax) return fail(FP8_ERR_INVALID, "g or amax is NULL");
  if (!aligned16(g)) return fail(FP8_ERR_INVALID, "g must be 16-byte aligned");
  if (n < 1 || n > (int64_t{1} << 40)) return fail(FP8_ERR_INVALID, "n %lld out of range", (long long)n);
  const int sms = current_sms();
  if (sms < 1) return fail(FP8_ERR_CUDA, "no CUDA device");
  return grad_launch(fp8lin::launch_grad_amax(g, n, amax, sms, as_stream(stream)), "grad amax launch");
}

fp8_status_t fp8_grad_quantize(const void* g, int64_t n, const float* amax, int32_t world, void* codes,
                               int64_t padded_n, float* scale, fp8_stream_t stream) {
  g_msg.clear();
  if (!g || !amax || !codes || !scale) return fail(FP8_ERR_INVALID, "g, amax, codes or scale is NULL");
  if (!aligned16(g) || !aligned16(codes)) return fail(FP8_ERR_INVALID, "g and codes must be 16-byte aligned");
  if (world < 1 || world > FP8_GRAD_MAX_WORLD) return fail(FP8_ERR_INVALID, "world %d out of range", world);
  if (n < 1 || n > (int64_t{1} << 40) || padded_n < n || padded_n > (int64_t{1} << 41))
    return fail(FP8_ERR_INVALID, "n %lld / padded_n %lld out of range", (long long)n, (long long)padded_n);
  const int sms = current_sms();
  if (sms < 1) return fail(FP8_ERR_CUDA, "no CUDA device");
  return grad_launch(fp8lin::launch_grad_quantize(g, n, amax, world, codes, padded_n, scale, sms, as_stream(stream)),
                     "grad quantize launch");
}

fp8_status_t fp8_grad_reduce(const void* recv, int32_t world, int64_t chunk, void* out, fp8_stream_t stream) {
  g_msg.clear();
  if (!recv || !out) return fail(FP8_ERR_INVALID, "recv or out is NULL");
  if (!aligned16(recv) || !aligned16(out)) return fail(FP8_ERR_INVALID, "recv and out must be 16-byte aligned");
  if (world < 1 || world > FP8_GRAD_MAX_WORLD) return fail(FP8_ERR_INVALID, "world %d out of range", world);
  if (chunk < 16 || chunk % 16 != 0 || chunk > (int64_t{1} << 40))
    return fail(FP8_ERR_INVALID, "chunk %lld must be a positive multiple of 16", (long long)chunk);
  const int sms = current_sms();
  if (sms < 1) return fail(FP8_ERR_CUDA, "no CUDA device");
  return grad_launch(fp8lin::launch_grad_reduce(recv, world, chunk, out, sms, as_stream(stream)), "grad reduce launch");
}

fp8_status_t fp8_grad_dequantize(const void* codes, int64_t n, const float* scale, int32_t world, int32_t average,
                                 void* out, fp8_stream_t stream) {
  g_msg.clear();
  if (!codes || !scale || !out) return fail(FP8_ERR_INVALID, "codes, scale or out is NULL");
  if (!aligned16(codes) || !aligned16(out)) return fail(FP8_ERR_INVALID, "codes and out must be 16-byte aligned");
  if (world < 1 || world > FP8_GRAD_MAX_WORLD) return fail(FP8_ERR_INVALID, "world %d out of range", world);
  if (n < 1 || n > (int64_t{1} << 40)) return fail(FP8_ERR_INVALID, "n %lld out of range", (long long)n);
  const int sms = current_sms();
  if (sms < 1) return fail(FP8_ERR_CUDA, "no CUDA device");
  return grad_launch(fp8lin::launch_grad_dequantize(codes, n, scale, world, average != 0 ? 1 : 0, out, sms,
                                                    as_stream(stream)),
                     "grad dequantize launch");
}

fp8_status_t fp8_update_scales(fp8_recipe_t* r, fp8_stream_t stream) {
  g_msg.clear();
  if (!r) return fail(FP8_ERR_INVALID, "recipe is NULL");
  cudaError_t e = fp8lin::launch_update_scales(r->dev, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "update_scales launch");
  return FP8_OK;
}

fp8_status_t fp8_get_state(fp8_recipe_t* r, int32_t tensor_id, fp8_tensor_state_t* state,
                           float* history, fp8_stream_t stream) {
  g_msg.clear();
  if (!r) return fail(FP8_ERR_INVALID, "recipe is NULL");
  if (fp8_status_t st = check_id(r, tensor_id, "tensor_id")) return st;
  if (!state) return fail(FP8_ERR_INVALID, "state is NULL");
  cudaStream_t s = as_stream(stream);
  const int H = r->dev.H;
  cudaError_t e = cudaMemcpyAsync(r->host_state, r->dev.states + tensor_id, sizeof(TensorState),
                                  cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(r->host_hist, r->dev.history + static_cast<int64_t>(tensor_id) * H,
                        sizeof(float) * H, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e, "copying state to host");
  if (fp8_status_t st = read_device_error(r, s)) return st;  // synchronises
  const TensorState& t = *r->host_state;
  auto bits = [](uint32_t b) {
    float f;
    memcpy(&f, &b, sizeof f);
    return f;
  };
  state->scale = t.scale;
  state->scale_inv = t.scale_inv;
  state->cast_scale = t.cast_scale;
  state->cast_scale_inv = t.cast_scale_inv;
  state->amax_pending = bits(t.amax_pending);
  state->amax_last = bits(t.amax_last);
  state->n_saturated = t.n_sat;
  state->n_underflow = t.n_und;
  state->n_saturated_last = t.n_sat_last;
  state->n_underflow_last = t.n_und_last;
  state->dtype = t.dtype;
  state->recorded = t.recorded;
  if (history) {
    for (int i = 0; i < H; ++i) history[i] = r->host_hist[(t.head + 1 + i) % H];  // oldest first
  }
  return FP8_OK;
}

fp8_status_t fp8_set_state(fp8_recipe_t* r, int32_t tensor_id, const float* history, float scale,
                           int32_t dtype, fp8_stream_t stream) {
  g_msg.clear();
  if (!r) return fail(FP8_ERR_INVALID, "recipe is NULL");
  if (fp8_status_t st = check_id(r, tensor_id, "tensor_id")) return st;
  if (!history) return fail(FP8_ERR_INVALID, "history is NULL");
  if (!valid_dtype(dtype)) return fail(FP8_ERR_INVALID, "unknown dtype %d", dtype);
  if (!(scale > 0.0f) || !std::isfinite(scale))
    return fail(FP8_ERR_INVALID, "scale must be finite and > 0");
  const int H = r->dev.H;
  for (int i = 0; i < H; ++i) {
    if (!(history[i] >= 0.0f) || !std::isfinite(history[i]))
      return fail(FP8_ERR_INVALID, "history[%d] must be finite and >= 0", i);
    r->host_hist[i] = history[i] == 0.0f ? 0.0f : history[i];  // -0 -> +0
  }
  cudaStream_t s = as_stream(stream);
  cudaError_t e = cudaMemcpyAsync(r->dev_hist_in, r->host_hist, sizeof(float) * H,
                                  cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = fp8lin::launch_set_state(r->dev, tensor_id, r->dev_hist_in, scale, dtype, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "set_state");
  return FP8_OK;
}

fp8_status_t fp8_debug_inject_stall(fp8_recipe_t* r, int32_t which) {
  g_msg.clear();
  if (!r) return fail(FP8_ERR_INVALID, "recipe is NULL");
  if (which != FP8_STALL_CAST && which != FP8_STALL_GEMM)
    return fail(FP8_ERR_INVALID, "unknown stall target %d", which);
  r->stall_once |= which == FP8_STALL_CAST ? 1u : 2u;
  return FP8_OK;
}

fp8_status_t fp8_check_device_error(fp8_recipe_t* r, fp8_stream_t stream) {
  g_msg.clear();
  if (!r) return fail(FP8_ERR_INVALID, "recipe is NULL");
  return read_device_error(r, as_stream(stream));
}

}  // extern "C"
