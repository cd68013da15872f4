"""CPU oracle for the scaled FP8 linear path (per-tensor and MX block scaling).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg import this package.  The product
library never does, and it shares no code with the CUDA path.

The arithmetic lives in ``fp8_oracle.c`` (fp64 where the pages leave precision
open); this module marshals numpy arrays into it and holds the delayed-scaling
recipe bookkeeping (``recipe.py``).  Page references:

* [TE] "4.2 Hopper I -- Transformer Engine / FP8" (aegloslab.com/nvidia/43),
  S4.2.3-S4.2.6.
* [LP] "FP8 and low-precision formats" (aiunderstanding.org), technical insight.
"""
import ctypes
import os

import numpy as np

from . import build as _build

E4M3 = 0
E5M2 = 1

_lib = None


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        if not _build.up_to_date():
            _build.build()
        L = ctypes.CDLL(_build.LIB)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        L.oracle_fp8_decode.argtypes = [ctypes.c_uint8, ctypes.c_int]
        L.oracle_fp8_decode.restype = ctypes.c_double
        L.oracle_fp8_max.argtypes = [ctypes.c_int]
        L.oracle_fp8_max.restype = ctypes.c_double
        L.oracle_fp8_encode.argtypes = [ctypes.c_float, ctypes.c_int]
        L.oracle_fp8_encode.restype = ctypes.c_uint8
        L.oracle_fp8_decode_array.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
        L.oracle_fp8_encode_array.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
        L.oracle_bf16_to_float.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_float.restype = ctypes.c_float
        L.oracle_double_to_bf16.argtypes = [ctypes.c_double]
        L.oracle_double_to_bf16.restype = ctypes.c_uint16
        L.oracle_double_to_bf16_array.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        L.oracle_amax_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64]
        L.oracle_amax_bf16.restype = ctypes.c_float
        L.oracle_cast_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int,
                                       ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint64),
                                       ctypes.POINTER(ctypes.c_uint64)]
        L.oracle_scale_from_amax.argtypes = [ctypes.c_float, ctypes.c_int, ctypes.c_float]
        L.oracle_scale_from_amax.restype = ctypes.c_float
        L.oracle_reciprocal.argtypes = [ctypes.c_float]
        L.oracle_reciprocal.restype = ctypes.c_float
        L.oracle_gemm_rows.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p,
                                       ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_float,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_set_num_threads.argtypes = [ctypes.c_int]
        L.oracle_fp8_encode_double.argtypes = [ctypes.c_double, ctypes.c_int]
        L.oracle_fp8_encode_double.restype = ctypes.c_uint8
        L.oracle_mx_scale_exponent.argtypes = [ctypes.c_double, ctypes.c_int]
        L.oracle_mx_scale_exponent.restype = ctypes.c_int
        L.oracle_e8m0_value.argtypes = [ctypes.c_uint8]
        L.oracle_e8m0_value.restype = ctypes.c_double
        L.oracle_mx_quantize.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_allreduce_scale.argtypes = [ctypes.c_float, ctypes.c_int]
        L.oracle_allreduce_scale.restype = ctypes.c_float
        L.oracle_allreduce_e5m2.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_mx_gemm_rows.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_cast_f32.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int,
                                      ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint64),
                                      ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_float)]
        L.oracle_gelu.argtypes = [ctypes.c_double]
        L.oracle_gelu.restype = ctypes.c_double
        L.oracle_dgelu.argtypes = [ctypes.c_double]
        L.oracle_dgelu.restype = ctypes.c_double
        L.oracle_gelu_array.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        L.oracle_dgelu_array.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        del u8p
        _lib = L
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads():
    return int(lib().oracle_num_threads())


def set_num_threads(n):
    """Threads of the oracle's later parallel loops (results do not depend on it)."""
    lib().oracle_set_num_threads(int(n))


def fp8_max(fmt):
    """Largest finite value of the format ([TE] S4.2.5 uses 448 for E4M3)."""
    return float(lib().oracle_fp8_max(fmt))


def decode(codes, fmt):
    """Exact value of each FP8 code (float64 array, NaN/Inf as IEEE)."""
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().oracle_fp8_decode_array(_ptr(c), c.size, fmt, _ptr(out))
    return out


def encode(values, fmt):
    """Saturating round-to-nearest-even encode of fp32 values."""
    v = _c(values, np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().oracle_fp8_encode_array(_ptr(v), v.size, fmt, _ptr(out))
    return out


def bf16_to_f32(bits):
    """Exact fp32 value of bf16 bit patterns (uint16 array)."""
    b = _c(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f64_to_bf16(y):
    """Round float64 values to bf16 bit patterns, nearest-even."""
    v = _c(y, np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().oracle_double_to_bf16_array(_ptr(v), v.size, _ptr(out))
    return out


def amax(x_bits):
    """max |x| of a bf16 tensor given as uint16 bit patterns ([TE] S4.2.4)."""
    x = _c(x_bits, np.uint16)
    return np.float32(lib().oracle_amax_bf16(_ptr(x), x.size))


def cast(x_bits, scale, fmt):
    """q = round_to_fp8(x * scale) with saturation ([TE] S4.2.4).

    Returns (codes uint8 same shape as x, n_saturated, n_underflow)."""
    x = _c(x_bits, np.uint16)
    q = np.empty(x.shape, dtype=np.uint8)
    ns = ctypes.c_uint64(0)
    nu = ctypes.c_uint64(0)
    lib().oracle_cast_bf16(_ptr(x), x.size, ctypes.c_float(float(np.float32(scale))), fmt, _ptr(q),
                           ctypes.byref(ns), ctypes.byref(nu))
    return q, int(ns.value), int(nu.value)


def cast_f32(values, scale, fmt):
    """The next stage's cast in a GEMM epilogue ([TE] S4.2.4, "composed with
    the next stage's scale"): codes of fp32(v * scale) for fp32 values v.

    Returns (codes uint8, n_saturated, n_underflow, amax = max|v| as fp32)."""
    v = _c(values, np.float32)
    q = np.empty(v.shape, dtype=np.uint8)
    ns = ctypes.c_uint64(0)
    nu = ctypes.c_uint64(0)
    am = ctypes.c_float(0.0)
    lib().oracle_cast_f32(_ptr(v), v.size, ctypes.c_float(float(np.float32(scale))), fmt, _ptr(q),
                          ctypes.byref(ns), ctypes.byref(nu), ctypes.byref(am))
    return q, int(ns.value), int(nu.value), np.float32(am.value)


def gelu(x):
    """GELU, tanh form, in fp64: the MLP activation of the transformer layer
    ([TE] S4.2.6's te.TransformerLayer; the function is a reading)."""
    v = _c(x, np.float64)
    out = np.empty(v.shape, dtype=np.float64)
    lib().oracle_gelu_array(_ptr(v), v.size, _ptr(out))
    return out


def dgelu(x):
    """Derivative of gelu() in fp64."""
    v = _c(x, np.float64)
    out = np.empty(v.shape, dtype=np.float64)
    lib().oracle_dgelu_array(_ptr(v), v.size, _ptr(out))
    return out


def scale_from_amax(m, fmt, prev_scale=1.0):
    """scale = FP8_MAX / m in fp32 ([TE] S4.2.4, S4.2.5)."""
    return np.float32(lib().oracle_scale_from_amax(ctypes.c_float(float(np.float32(m))), fmt,
                                                   ctypes.c_float(float(np.float32(prev_scale)))))


def reciprocal(s):
    """1/scale in fp32 -- the dequantisation multiplier ([TE] S4.2.4)."""
    return np.float32(lib().oracle_reciprocal(ctypes.c_float(float(np.float32(s)))))


def gemm(A, afmt, B, bfmt, factor, rows=None, want_abs=True, want_bf16=True):
    """Dequantised FP8 GEMM D = (A . B^T) * factor on codes, fp64 accumulation.

    A: uint8 [M, K]; B: uint8 [N, K]; factor: the fp32 product of the two
    operands' 1/scale.  ``rows`` selects output rows (all when None).
    Returns (acc float64 [R, N], absacc float64 [R, N] or None, bf16 bits [R, N] or None).
    """
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    if rows is None:
        R = M
        rp = None
        rows_arr = None
    else:
        rows_arr = _c(rows, np.int64)
        assert rows_arr.size == 0 or (rows_arr.min() >= 0 and rows_arr.max() < M)
        R = rows_arr.size
        rp = _ptr(rows_arr)
    acc = np.empty((R, N), dtype=np.float64)
    ab = np.empty((R, N), dtype=np.float64) if want_abs else None
    out = np.empty((R, N), dtype=np.uint16) if want_bf16 else None
    lib().oracle_gemm_rows(_ptr(A), afmt, K, _ptr(B), bfmt, K, M, N, K, rp, R,
                           ctypes.c_float(float(np.float32(factor))), _ptr(acc),
                           _ptr(ab) if ab is not None else None,
                           _ptr(out) if out is not None else None)
    return acc, ab, out


def encode_double(v, fmt):
    """Saturating RNE encode of one exact (double) value."""
    return int(lib().oracle_fp8_encode_double(float(v), fmt))


# --------------------------------------------------------------------------
# Block scaling, MX style ([LP] format overview: per-tensor or per-block scale
# factors; MXFP8 elements share one power-of-two scale per block of 32).


def mx_scale_exponent(amax_value, fmt):
    """k with block scale 2^-k: the largest k in [-127, 127] such that
    amax * 2^k <= FP8_MAX (-127 when there is none)."""
    return int(lib().oracle_mx_scale_exponent(float(amax_value), fmt))


def e8m0_value(code):
    """Value of an E8M0 scale code, 2^(code-127) (0xFF is NaN)."""
    return float(lib().oracle_e8m0_value(int(code)))


def mx_quantize(x_bits, fmt):
    """MX quantisation of a bf16 matrix along its rows.

    x_bits: uint16 [rows, cols].  Returns (codes uint8 [rows, cols], scale
    codes uint8 [rows, ceil(cols/32)])."""
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    sc = np.empty((rows, (cols + 31) // 32), dtype=np.uint8)
    lib().oracle_mx_quantize(_ptr(x), rows, cols, fmt, _ptr(q), _ptr(sc))
    return q, sc


def mx_gemm(A, afmt, sa, B, bfmt, sb, rows=None, want_abs=True, want_bf16=True):
    """D = dequant(A) . dequant(B)^T for MX operands, fp64 accumulation.

    A: uint8 [M, K], sa: uint8 [M, ceil(K/32)]; B: uint8 [N, K], sb: uint8
    [N, ceil(K/32)].  Returns (acc, absacc or None, bf16 bits or None) for the
    selected rows (all when None)."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    nb = (K + 31) // 32
    sa = _c(sa, np.uint8)
    sb = _c(sb, np.uint8)
    assert sa.shape == (M, nb) and sb.shape == (N, nb)
    if rows is None:
        R, rp = M, None
    else:
        rows_arr = _c(rows, np.int64)
        assert rows_arr.size == 0 or (rows_arr.min() >= 0 and rows_arr.max() < M)
        R, rp = rows_arr.size, _ptr(rows_arr)
    acc = np.empty((R, N), dtype=np.float64)
    ab = np.empty((R, N), dtype=np.float64) if want_abs else None
    out = np.empty((R, N), dtype=np.uint16) if want_bf16 else None
    lib().oracle_mx_gemm_rows(_ptr(A), afmt, _ptr(sa), _ptr(B), bfmt, _ptr(sb), M, N, K, rp, R, _ptr(acc),
                              _ptr(ab) if ab is not None else None,
                              _ptr(out) if out is not None else None)
    return acc, ab, out


# --------------------------------------------------------------------------
# FP8 gradient all-reduce with automatic scaling ([LP] use cases: E5M2 for
# gradient communication; [FL]: automatic scaling during the all-reduce).


def allreduce_scale(amax_value, world):
    """Shared scale 57344 / fp32(world * amax) (fp32; 1 for amax 0/non-finite)."""
    return np.float32(lib().oracle_allreduce_scale(ctypes.c_float(float(np.float32(amax_value))), int(world)))


def allreduce_e5m2(grads_bits, average=False):
    """All-reduce of world bf16 gradients through E5M2.

    grads_bits: uint16 [world, n].  Returns (out bf16 bits [n], reduced codes
    uint8 [n], (s, 1/s) as float32)."""
    g = _c(grads_bits, np.uint16)
    world, n = g.shape
    out = np.empty(n, dtype=np.uint16)
    codes = np.empty(n, dtype=np.uint8)
    sc = np.empty(2, dtype=np.float32)
    lib().oracle_allreduce_e5m2(_ptr(g), world, n, 1 if average else 0, _ptr(out), _ptr(codes), _ptr(sc))
    return out, codes, (sc[0], sc[1])


from .recipe import DelayedRecipe, TensorState  # noqa: E402,F401
