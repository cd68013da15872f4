"""Per-tensor, dynamically scaled FP8 linear layer for GB300 (sm_103a).

Python binding of ``libfp8lin.so`` (C ABI in ``include/fp8lin.h``).  This
module only marshals arguments: every step of the path -- amax, scale, cast,
GEMM, history update -- runs in the library's CUDA kernels.  There is no CPU
fallback: if the library is not built, every call raises.

The functions keep the C names (``fp8_recipe_create``, ``fp8_amax_quantize``,
``fp8_gemm``, ``fp8_update_scales``, ...).  Buffers may be given as torch CUDA
tensors or raw device addresses (ints); ``stream`` may be None (torch's current
stream), a ``torch.cuda.Stream`` or a raw ``cudaStream_t`` int.  ``Recipe`` is a
small convenience wrapper that allocates outputs with torch.

Method: "4.2 Hopper I -- Transformer Engine / FP8" (aegloslab.com/nvidia/43),
S4.2.4 (amax, scale = FP8_MAX/amax, scaled cast, FP32-accumulated GEMM with
1/scale dequantisation, delayed scaling with an amax history) and S4.2.6
(HYBRID format, history length 16, "max" rule).
"""
import ctypes
import os

from .build import LIB as _LIB_PATH

E4M3 = 0
E5M2 = 1
RECIPE_HYBRID = 0
RECIPE_E4M3 = 1
AMAX_MAX = 0
AMAX_MOST_RECENT = 1
DELAYED = 0
CURRENT = 1
OUT_BF16 = 0
OUT_F32 = 1
OUT_E4M3 = 2
OUT_E5M2 = 3
K_MAJOR = 0    # GEMM operand stored [M or N, K]
MN_MAJOR = 1   # GEMM operand stored [K, M or N]
ACT_NONE = 0   # epilogue activation: none
ACT_GELU = 1   # gelu(y) stored; aux <- bf16(gelu'(y))
ACT_DGELU = 2  # y * aux stored (aux: the forward's gelu')

FP8_MAX = {E4M3: 448.0, E5M2: 57344.0}

STATUS = {0: "FP8_OK", 1: "FP8_ERR_INVALID", 2: "FP8_ERR_UNSUPPORTED", 3: "FP8_ERR_CUDA",
          4: "FP8_ERR_TIMEOUT", 5: "FP8_ERR_NOMEM"}

# C symbols the header declares (checked by the CPU test of the ABI).
EXPORTS = ("fp8_recipe_create", "fp8_recipe_destroy", "fp8_amax_quantize", "fp8_gemm", "fp8_gemm_layout",
           "fp8_gemm_act",
           "fp8_update_scales", "fp8_get_state", "fp8_set_state", "fp8_check_device_error",
           "fp8_status_string", "fp8_last_error_message", "fp8_quantize_current_noalloc",
           "fp8_mx_scale_bytes", "fp8_mx_quantize", "fp8_mx_gemm",
           "fp8_grad_amax", "fp8_grad_quantize", "fp8_grad_reduce", "fp8_grad_dequantize",
           "fp8_debug_inject_stall")

# Largest n fp8_quantize_current_noalloc accepts (its static scratch covers this much).
NOALLOC_MAX_ELEMENTS = 1 << 30

# Largest world size of the FP8 gradient all-reduce steps.
GRAD_MAX_WORLD = 32768


class Fp8Error(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class TensorStateC(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_float), ("scale_inv", ctypes.c_float),
                ("cast_scale", ctypes.c_float), ("cast_scale_inv", ctypes.c_float),
                ("amax_pending", ctypes.c_float), ("amax_last", ctypes.c_float),
                ("n_saturated", ctypes.c_uint64), ("n_underflow", ctypes.c_uint64),
                ("n_saturated_last", ctypes.c_uint64), ("n_underflow_last", ctypes.c_uint64),
                ("dtype", ctypes.c_int32), ("recorded", ctypes.c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


_lib = None


def library_path():
    return _LIB_PATH


def load():
    """Load libfp8lin.so (raises if it was not built -- no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it first "
                           "(python -m fp8_mixed_precision_history_gb300.build)")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    L.fp8_recipe_create.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, vp]
    L.fp8_recipe_destroy.argtypes = [vp]
    L.fp8_amax_quantize.argtypes = [vp, i32, vp, i64, i64, i32, i32, i32, vp, vp, vp]
    L.fp8_gemm.argtypes = [vp, i32, vp, i32, i64, i32, vp, i32, i64, i64, i64, i64, vp, i32, i64,
                           i32, vp]
    L.fp8_gemm_layout.argtypes = [vp, i32, vp, i32, i32, i64, i32, vp, i32, i32, i64, i64, i64, i64, vp, i32,
                                  i64, i32, vp]
    L.fp8_gemm_act.argtypes = [vp, i32, vp, i32, i32, i64, i32, vp, i32, i32, i64, i64, i64, i64, vp, i32,
                               i64, i32, i32, vp, i64, vp]
    L.fp8_update_scales.argtypes = [vp, vp]
    L.fp8_get_state.argtypes = [vp, i32, ctypes.POINTER(TensorStateC), ctypes.POINTER(ctypes.c_float), vp]
    L.fp8_set_state.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_float), ctypes.c_float, i32, vp]
    L.fp8_check_device_error.argtypes = [vp, vp]
    L.fp8_quantize_current_noalloc.argtypes = [vp, i64, i32, vp, vp, vp, vp]
    L.fp8_mx_scale_bytes.argtypes = [i64, i64]
    L.fp8_mx_scale_bytes.restype = i64
    L.fp8_mx_quantize.argtypes = [vp, vp, i64, i64, i32, vp, vp, vp, vp, vp]
    L.fp8_mx_gemm.argtypes = [vp, vp, i32, i64, vp, vp, i32, i64, vp, i64, i64, i64, vp, i32, i64, vp]
    L.fp8_grad_amax.argtypes = [vp, i64, vp, vp]
    L.fp8_grad_quantize.argtypes = [vp, i64, vp, i32, vp, i64, vp, vp]
    L.fp8_grad_reduce.argtypes = [vp, i32, i64, vp, vp]
    L.fp8_grad_dequantize.argtypes = [vp, i64, vp, i32, i32, vp, vp]
    L.fp8_debug_inject_stall.argtypes = [vp, i32]
    L.fp8_status_string.argtypes = [ctypes.c_int]
    L.fp8_status_string.restype = ctypes.c_char_p
    L.fp8_last_error_message.argtypes = []
    L.fp8_last_error_message.restype = ctypes.c_char_p
    for name in ("fp8_recipe_create", "fp8_recipe_destroy", "fp8_amax_quantize", "fp8_gemm",
                 "fp8_gemm_layout", "fp8_gemm_act", "fp8_update_scales", "fp8_get_state", "fp8_set_state", "fp8_check_device_error",
                 "fp8_quantize_current_noalloc", "fp8_mx_quantize", "fp8_mx_gemm", "fp8_grad_amax",
                 "fp8_grad_quantize", "fp8_grad_reduce", "fp8_grad_dequantize", "fp8_debug_inject_stall"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st):
    if st != 0:
        msg = load().fp8_last_error_message().decode(errors="replace")
        raise Fp8Error(st, msg)


# ------------------------------------------------------------- C names ----

def fp8_status_string(status):
    return load().fp8_status_string(int(status)).decode()


def fp8_last_error_message():
    return load().fp8_last_error_message().decode(errors="replace")


def fp8_recipe_create(format=RECIPE_HYBRID, amax_history_len=16, algo=AMAX_MAX, num_tensors=1,
                      stream=None):
    h = ctypes.c_void_p()
    _check(load().fp8_recipe_create(ctypes.byref(h), format, amax_history_len, algo, num_tensors,
                                    _stream(stream)))
    return h.value


def fp8_recipe_destroy(r):
    _check(load().fp8_recipe_destroy(r))


def fp8_amax_quantize(r, tensor_id, x, rows, cols, dtype, mode, update_now, out, out_t=None,
                      stream=None):
    _check(load().fp8_amax_quantize(r, tensor_id, _ptr(x), rows, cols, dtype, mode,
                                    1 if update_now else 0, _ptr(out), _ptr(out_t), _stream(stream)))


def fp8_gemm(r, a_id, A, a_dtype, lda, b_id, B, b_dtype, ldb, M, N, K, D, d_dtype, ldd,
             amax_out_id=-1, stream=None):
    _check(load().fp8_gemm(r, a_id, _ptr(A), a_dtype, lda, b_id, _ptr(B), b_dtype, ldb, M, N, K,
                           _ptr(D), d_dtype, ldd, amax_out_id, _stream(stream)))


def fp8_gemm_layout(r, a_id, A, a_dtype, a_major, lda, b_id, B, b_dtype, b_major, ldb, M, N, K, D, d_dtype,
                    ldd, amax_out_id=-1, stream=None):
    _check(load().fp8_gemm_layout(r, a_id, _ptr(A), a_dtype, a_major, lda, b_id, _ptr(B), b_dtype, b_major,
                                  ldb, M, N, K, _ptr(D), d_dtype, ldd, amax_out_id, _stream(stream)))


def fp8_gemm_act(r, a_id, A, a_dtype, a_major, lda, b_id, B, b_dtype, b_major, ldb, M, N, K, D, d_dtype, ldd,
                 amax_out_id=-1, act=ACT_NONE, aux=None, ld_aux=0, stream=None):
    _check(load().fp8_gemm_act(r, a_id, _ptr(A), a_dtype, a_major, lda, b_id, _ptr(B), b_dtype, b_major, ldb,
                               M, N, K, _ptr(D), d_dtype, ldd, amax_out_id, act, _ptr(aux), ld_aux,
                               _stream(stream)))


def fp8_update_scales(r, stream=None):
    _check(load().fp8_update_scales(r, _stream(stream)))


def fp8_get_state(r, tensor_id, history_len, stream=None):
    """Returns (state dict, history list oldest first)."""
    st = TensorStateC()
    h = (ctypes.c_float * history_len)()
    _check(load().fp8_get_state(r, tensor_id, ctypes.byref(st), h, _stream(stream)))
    return st.as_dict(), [float(v) for v in h]


def fp8_set_state(r, tensor_id, history, scale, dtype, stream=None):
    h = (ctypes.c_float * len(history))(*[float(v) for v in history])
    _check(load().fp8_set_state(r, tensor_id, h, float(scale), dtype, _stream(stream)))


def fp8_check_device_error(r, stream=None):
    _check(load().fp8_check_device_error(r, _stream(stream)))


def fp8_quantize_current_noalloc(x, n, dtype, out, scale_out, counts_out=None, stream=None):
    """Current-scaling cast that allocates no device memory (for callers that
    cannot allocate while they run, e.g. inside a framework that owns all device
    memory).  Its scratch is a static array inside the library, shared by all
    calls on a GPU: do not overlap calls on unordered streams.  scale_out gets
    {scale, 1/scale} (2 floats), counts_out {#saturated, #underflowed} (2 x
    64-bit) or is None."""
    _check(load().fp8_quantize_current_noalloc(_ptr(x), n, dtype, _ptr(out), _ptr(scale_out),
                                               _ptr(counts_out), _stream(stream)))


def fp8_mx_scale_bytes(rows, cols):
    """Bytes of the block-scale array of an MX [rows, cols] matrix."""
    return int(load().fp8_mx_scale_bytes(rows, cols))


def fp8_mx_quantize(r, x, rows, cols, dtype, q, q_scale, q_t=None, q_t_scale=None, stream=None):
    _check(load().fp8_mx_quantize(r, _ptr(x), rows, cols, dtype, _ptr(q), _ptr(q_scale), _ptr(q_t),
                                  _ptr(q_t_scale), _stream(stream)))


def fp8_mx_gemm(r, A, a_dtype, lda, a_scale, B, b_dtype, ldb, b_scale, M, N, K, D, d_dtype, ldd,
                stream=None):
    _check(load().fp8_mx_gemm(r, _ptr(A), a_dtype, lda, _ptr(a_scale), _ptr(B), b_dtype, ldb, _ptr(b_scale),
                              M, N, K, _ptr(D), d_dtype, ldd, _stream(stream)))


def fp8_grad_amax(g, n, amax, stream=None):
    _check(load().fp8_grad_amax(_ptr(g), n, _ptr(amax), _stream(stream)))


def fp8_grad_quantize(g, n, amax, world, codes, padded_n, scale, stream=None):
    _check(load().fp8_grad_quantize(_ptr(g), n, _ptr(amax), world, _ptr(codes), padded_n, _ptr(scale),
                                    _stream(stream)))


def fp8_grad_reduce(recv, world, chunk, out, stream=None):
    _check(load().fp8_grad_reduce(_ptr(recv), world, chunk, _ptr(out), _stream(stream)))


def fp8_grad_dequantize(codes, n, scale, world, average, out, stream=None):
    _check(load().fp8_grad_dequantize(_ptr(codes), n, _ptr(scale), world, 1 if average else 0, _ptr(out),
                                      _stream(stream)))


STALL_CAST = 0
STALL_GEMM = 1


def fp8_debug_inject_stall(r, which):
    """Test hook: the next launch of the chosen kernel on this recipe times out
    on purpose (bounded wait), so that failure reporting can be checked."""
    _check(load().fp8_debug_inject_stall(r, which))


# ------------------------------------------------------------ wrapper ----

class Recipe:
    """A recipe handle plus torch-allocated outputs (plumbing only)."""

    def __init__(self, num_tensors, amax_history_len=16, algo=AMAX_MAX, format=RECIPE_HYBRID,
                 stream=None):
        self.H = amax_history_len
        self.handle = fp8_recipe_create(format, amax_history_len, algo, num_tensors, stream)

    def close(self):
        if self.handle:
            fp8_recipe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def quantize(self, tensor_id, x, dtype, mode=DELAYED, update_now=False, transpose=False,
                 out=None, out_t=None, stream=None):
        import torch

        rows, cols = (x.shape[0], x[0].numel()) if x.dim() > 1 else (1, x.numel())
        if out is None:
            out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
        if transpose and out_t is None:
            out_t = torch.empty((cols, rows), dtype=torch.uint8, device=x.device)
        fp8_amax_quantize(self.handle, tensor_id, x, rows, cols, dtype, mode, update_now, out,
                          out_t if transpose else None, stream)
        return (out, out_t) if transpose else out

    def gemm(self, a_id, A, a_dtype, b_id, B, b_dtype, out_dtype=OUT_BF16, out=None,
             amax_out_id=-1, stream=None, a_major=K_MAJOR, b_major=K_MAJOR, act=ACT_NONE, aux=None):
        """D = A B^T dequantised.  K_MAJOR operands are [M, K] / [N, K];
        MN_MAJOR operands are stored [K, M] / [K, N].  act / aux: the epilogue
        activation (fp8_gemm_act); aux is a bf16 [M, N] tensor."""
        import torch

        M, K = A.shape if a_major == K_MAJOR else A.shape[::-1]
        N = B.shape[0] if b_major == K_MAJOR else B.shape[1]
        if out is None:
            dt = {OUT_F32: torch.float32, OUT_BF16: torch.bfloat16}.get(out_dtype, torch.uint8)
            out = torch.empty((M, N), dtype=dt, device=A.device)
        fp8_gemm_act(self.handle, a_id, A, a_dtype, a_major, A.stride(0), b_id, B, b_dtype, b_major,
                     B.stride(0), M, N, K, out, out_dtype, out.stride(0), amax_out_id, act, aux,
                     aux.stride(0) if aux is not None else 0, stream)
        return out

    def mx_quantize(self, x, dtype, transpose=False, stream=None):
        """MX block quantisation of a bf16 [rows, cols] tensor.  Returns
        (q, q_scale) or (q, q_scale, q_t, q_t_scale); the scales are uint8
        arrays in the atom layout of the C header."""
        import torch

        rows, cols = x.shape
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
        qs = torch.empty(fp8_mx_scale_bytes(rows, cols), dtype=torch.uint8, device=x.device)
        qt = qts = None
        if transpose:
            qt = torch.empty((cols, rows), dtype=torch.uint8, device=x.device)
            qts = torch.empty(fp8_mx_scale_bytes(cols, rows), dtype=torch.uint8, device=x.device)
        fp8_mx_quantize(self.handle, x, rows, cols, dtype, q, qs, qt, qts, stream)
        return (q, qs, qt, qts) if transpose else (q, qs)

    def mx_gemm(self, A, a_dtype, a_scale, B, b_dtype, b_scale, out_dtype=OUT_BF16, out=None, stream=None):
        """D = dequant(A) . dequant(B)^T for MX operands (codes + atom scales)."""
        import torch

        M, K = A.shape
        N = B.shape[0]
        if out is None:
            dt = torch.float32 if out_dtype == OUT_F32 else torch.bfloat16
            out = torch.empty((M, N), dtype=dt, device=A.device)
        fp8_mx_gemm(self.handle, A, a_dtype, A.stride(0), a_scale, B, b_dtype, B.stride(0), b_scale, M, N, K,
                    out, out_dtype, out.stride(0), stream)
        return out

    def update_scales(self, stream=None):
        fp8_update_scales(self.handle, stream)

    def get_state(self, tensor_id, stream=None):
        return fp8_get_state(self.handle, tensor_id, self.H, stream)

    def set_state(self, tensor_id, history, scale, dtype, stream=None):
        fp8_set_state(self.handle, tensor_id, history, scale, dtype, stream)

    def check_device_error(self, stream=None):
        fp8_check_device_error(self.handle, stream)
