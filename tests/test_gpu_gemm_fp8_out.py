"""GEMM with the next stage's scale composed into the epilogue ("4.2 Hopper I
-- Transformer Engine / FP8", S4.2.4: the FP32 result is multiplied by 1/scale
"or composed with the next stage's scale").

With d_dtype FP8_OUT_E4M3 / FP8_OUT_E5M2 the kernel stores
D = round_to_fp8(y * s_out), y = fp32(acc * sinv_A * sinv_B), using the output
tensor's delayed scale, and records that tensor's max|y|, saturation and
underflow counts and cast scale.  Checked against:
* the same kernel's fp32 output y, cast with torch's float8 conversion
  (saturated first): bit for bit;
* the oracle's fp64 product scaled: each code the rounding of a value inside
  the fp32 accumulation bound (1e-6 * sum|ab|, scaled), and within one code
  step of the oracle's own encoding wherever that bound is below half a code
  spacing (a heavily cancelling sum can sit further while inside the bound);
* the recorded state: amax and counts recomputed from y, bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import f32_bits, to_host_u8

pytestmark = pytest.mark.gpu

MAX = {2: 448.0, 3: 57344.0}
UND = {2: 2.0 ** -10, 3: 2.0 ** -17}
TORCH_FP8 = {2: torch.float8_e4m3fn, 3: torch.float8_e5m2}
ORACLE_FMT = {2: oracle.E4M3, 3: oracle.E5M2}


def _tensor_codes(rng, shape, fmt):
    if fmt == 0:
        v = rng.standard_normal(shape) * (448.0 / 4.5)
    else:
        mag = np.exp(rng.uniform(np.log(1e-6), np.log(1e-1), shape)) * (57344.0 / 0.1)
        v = np.where(rng.random(shape) < 0.5, -mag, mag)
    return oracle.encode(v.astype(np.float32), fmt)


def _fp8_spacing(v, out):
    """Distance between neighbouring FP8 values around |v| (E4M3: 3 mantissa
    bits, subnormal step 2^-9; E5M2: 2 bits, 2^-16)."""
    mbits, sub = (3, 2.0 ** -9) if out == 2 else (2, 2.0 ** -16)
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, sub)))
    return np.maximum(np.exp2(e - mbits), sub)


def _ordered(codes, fmt):
    """FP8 codes -> integers ordered like their values (+0 == -0)."""
    c = np.asarray(codes).astype(np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


@pytest.mark.parametrize("out", [2, 3])
@pytest.mark.parametrize("shape", [(256, 512, 512), (129, 264, 144), (300, 1000, 208),
                                   (1024, 1024, 4096), (64, 512, 32)])
def test_fp8_output_matches_cast_of_fp32_output(gpu_lib, out, shape):
    fp8 = gpu_lib
    M, N, K = shape
    rng = np.random.default_rng(M + 7 * N + 13 * K + out)
    afmt, bfmt = (0, 0) if out == 2 else (1, 0)
    A = _tensor_codes(rng, (M, K), afmt)
    B = _tensor_codes(rng, (N, K), bfmt)
    sa, sb = (1.0 / 64, 1.0 / 256)
    R = fp8.Recipe(3)
    R.set_state(0, [1.0] * 16, sa, afmt)
    R.set_state(1, [1.0] * 16, sb, bfmt)
    # output scale chosen so that some values saturate and some underflow
    Ad = torch.from_numpy(A).cuda()
    Bd = torch.from_numpy(B).cuda()
    y32 = R.gemm(0, Ad, afmt, 1, Bd, bfmt, out_dtype=fp8.OUT_F32)
    ymax = float(y32.abs().max())
    s_out = float(np.float32(MAX[out] / (0.5 * ymax)))
    R.set_state(2, [0.5] * 16, s_out, out - 2)
    D8 = R.gemm(0, Ad, afmt, 1, Bd, bfmt, out_dtype=out, amax_out_id=2)
    torch.cuda.synchronize()
    R.check_device_error()

    # 1. the same kernel's fp32 output, cast with torch (saturating first)
    p = y32 * torch.tensor(s_out, dtype=torch.float32, device="cuda")
    want = p.clamp(-MAX[out], MAX[out]).to(TORCH_FP8[out]).view(torch.uint8)
    assert torch.equal(D8, want), f"{int((D8 != want).sum())} codes differ from the cast of y"

    # 2. the oracle: fp64 product, scaled.  A code must be the rounding of a
    # value inside the fp32 accumulation bound (1e-6 * sum|ab|, scaled), i.e.
    # within bound + one FP8 spacing; where that bound is below half a spacing,
    # within one code step of the oracle's own encoding.
    st0, _ = R.get_state(0)
    st1, _ = R.get_state(1)
    factor = np.float32(st0["cast_scale_inv"]) * np.float32(st1["cast_scale_inv"])
    acc, absacc, _ = oracle.gemm(A, afmt, B, bfmt, factor, want_bf16=False)
    yref = acc * float(factor)
    pref = np.clip(yref * s_out, -MAX[out], MAX[out])
    bound = 1e-6 * absacc * float(factor) * s_out
    dec = D8.cpu().view(TORCH_FP8[out]).double().numpy()
    sp = _fp8_spacing(np.maximum(np.abs(pref), np.abs(dec)), out)
    bad = np.abs(dec - pref) > bound + sp
    assert not bad.any(), f"{int(bad.sum())} codes beyond bound + one spacing"
    cref = oracle.encode(pref.astype(np.float32), ORACLE_FMT[out])
    tight = bound <= 0.5 * _fp8_spacing(np.abs(pref), out)
    d = np.abs(_ordered(to_host_u8(D8), out) - _ordered(cref, out))[tight]
    assert d.size and d.max() <= 1, f"codes up to {d.max()} steps from the oracle where the bound is tight"

    # 3. the output tensor's recorded state
    st, _ = R.get_state(2)
    yh = y32.cpu().numpy()
    ph = (yh.astype(np.float32) * np.float32(s_out)).astype(np.float32)
    assert f32_bits(st["amax_pending"]) == f32_bits(np.max(np.abs(yh)))
    assert st["n_saturated"] == int(np.sum(np.abs(ph) > MAX[out]))
    assert st["n_underflow"] == int(np.sum((yh != 0) & (np.abs(ph) <= UND[out])))
    assert st["n_saturated"] > 0
    assert f32_bits(st["cast_scale"]) == f32_bits(np.float32(s_out))
    assert f32_bits(st["cast_scale_inv"]) == f32_bits(oracle.reciprocal(s_out))
    assert st["dtype"] == out - 2 and st["recorded"] == 1
    # the oracle's amax agrees within the fp32 accumulation bound
    assert abs(float(st["amax_pending"]) - np.max(np.abs(yref))) <= 1e-6 * float(absacc.max() * factor)
    R.close()


def test_fp8_output_feeds_the_next_gemm(gpu_lib):
    """A GEMM consuming the FP8 output dequantises it with the output tensor's
    recorded 1/scale: chained result equals (decoded codes / s_out) . W2^T."""
    fp8 = gpu_lib
    rng = np.random.default_rng(5)
    M, K1, N1, N2 = 256, 512, 384, 256
    X = _tensor_codes(rng, (M, K1), 0)
    W1 = _tensor_codes(rng, (N1, K1), 0)
    W2 = _tensor_codes(rng, (N2, N1), 0)
    R = fp8.Recipe(4)
    R.set_state(0, [1.0] * 16, 1.0 / 64, 0)
    R.set_state(1, [1.0] * 16, 1.0 / 256, 0)
    R.set_state(3, [1.0] * 16, 1.0 / 256, 0)
    y = R.gemm(0, torch.from_numpy(X).cuda(), 0, 1, torch.from_numpy(W1).cuda(), 0, out_dtype=fp8.OUT_F32)
    s_out = float(np.float32(448.0 / float(y.abs().max())))
    R.set_state(2, [1.0] * 16, s_out, 0)
    Y8 = R.gemm(0, torch.from_numpy(X).cuda(), 0, 1, torch.from_numpy(W1).cuda(), 0,
                out_dtype=fp8.OUT_E4M3, amax_out_id=2)
    Z = R.gemm(2, Y8, 0, 3, torch.from_numpy(W2).cuda(), 0, out_dtype=fp8.OUT_F32)
    torch.cuda.synchronize()
    yq = Y8.cpu().view(torch.float8_e4m3fn).double() / np.float32(s_out)
    w2 = torch.from_numpy(W2).view(torch.float8_e4m3fn).double() * 256.0
    want = (yq @ w2.T).numpy()
    err = np.abs(Z.cpu().numpy() - want)
    scale = (yq.abs() @ w2.abs().T).numpy()
    assert np.all(err <= 1e-5 * scale + 1e-30)
    R.close()


def test_fp8_output_argument_checks(gpu_lib):
    fp8 = gpu_lib
    R = fp8.Recipe(3)
    A = torch.zeros((16, 32), dtype=torch.uint8, device="cuda")
    with pytest.raises(fp8.Fp8Error):
        R.gemm(0, A, 0, 1, A, 0, out_dtype=fp8.OUT_E4M3)  # no output tensor id
    R.close()
    R = fp8.Recipe(3, format=fp8.RECIPE_E4M3)
    with pytest.raises(fp8.Fp8Error):
        R.gemm(0, A, 0, 1, A, 0, out_dtype=fp8.OUT_E5M2, amax_out_id=2)
    R.close()
