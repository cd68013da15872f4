"""GEMM with the MLP's activation fused into the epilogue (fp8_gemm_act).

"4.2 Hopper I -- Transformer Engine / FP8", S4.2.4: the FP32 result is
multiplied by 1/scale "or composed with the next stage's scale"; S4.2.6's
te.TransformerLayer puts an activation between FC1 and FC2 (GELU, tanh form:
the reading taken).  FC1's forward stores gelu(y) -- as FC2's E4M3 operand --
and bf16(y) for the backward; FC2's dgrad stores y * gelu'(h) -- as FC1's E5M2
output gradient.

Checked, for every output of every shape:
* the fp32 value v the kernel stores (FP8_OUT_F32) against the oracle's fp64
  chain: y = exact sum * factor, v = gelu(y) or y * gelu'(h), within the
  propagated GEMM bound plus the fp32 evaluation error of the activation
  (derived in _act_bound);
* bf16 outputs equal RN(v) of the same kernel, bit for bit;
* FP8 outputs equal the oracle's epilogue cast of that fp32 v
  (oracle.cast_f32: the decision taken in the kernel's precision), bit for
  bit, and the output tensor's recorded amax, counts and cast scale equal the
  oracle's from the same values;
* the aux output bf16(y) equals RN of the same kernel's plain fp32 product.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import f32_bits, to_host_u16, to_host_u8
from test_gpu_gemm import _device_operand, _tensor_codes

pytestmark = pytest.mark.gpu

SHAPES = [(256, 512, 512), (129, 264, 144), (300, 1000, 208), (64, 512, 32), (1024, 1024, 4096),
          (384, 2048, 2048), (200, 136, 4112)]


def _bf16_rn(v32):
    return torch.from_numpy(np.ascontiguousarray(v32, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def _act_bound(y64, bound_y, act, h=None):
    """|v_gpu - v_oracle| for v = gelu(y) or y * gelu'(h).
    The GEMM leaves |y32 - y64| <= bound_y; |gelu'| <= 1.2 everywhere, so gelu
    moves it by at most 1.2 bound_y.  The fp32 evaluation (about six roundings
    of 2^-24, and tanhf within 2 ulp) adds at most 2^-20 (|x| + |gelu(x)|)
    for gelu, and 2^-20 (1 + |x| c (1 + 3a x^2)) for gelu' (1 - t^2 loses t's
    absolute error, amplified by the x c (1 + 3a x^2) term), then one rounding
    of the product y * gelu'(h)."""
    if act == 1:
        return 1.2 * bound_y + 2.0 ** -20 * (np.abs(y64) + np.abs(oracle.gelu(y64)))
    dg = oracle.dgelu(h)
    x = np.abs(h)
    ev = 2.0 ** -20 * (1.0 + x * 0.8 * (1.0 + 0.135 * x * x))
    return np.abs(dg) * bound_y + np.abs(y64) * ev + 2.0 ** -23 * np.abs(y64 * dg)


def _run(fp8, M, N, K, act, out_fmt, seed, a_major=0, b_major=0):
    """One activation GEMM in every output type; returns what the checks need."""
    rng = np.random.default_rng(seed)
    afmt = 0 if act == fp8.ACT_GELU else 1  # forward: E4M3 x E4M3; dgrad: E5M2 x E4M3
    A = _tensor_codes(rng, (M, K), afmt)
    B = _tensor_codes(rng, (N, K), 0)
    R = fp8.Recipe(3)
    R.set_state(0, [1.0] * 16, 1.0 / 64, afmt)
    R.set_state(1, [1.0] * 16, 1.0 / 256, 0)
    Av, Bv = _device_operand(A, a_major, None), _device_operand(B, b_major, None)
    kw = dict(a_major=a_major, b_major=b_major)
    y32 = R.gemm(0, Av, afmt, 1, Bv, 0, out_dtype=fp8.OUT_F32, **kw)
    h = None
    if act == fp8.ACT_DGELU:  # the forward's pre-activation: bf16 values around the GELU's bend
        h = torch.from_numpy((rng.standard_normal((M, N)) * 1.5).astype(np.float32)).to(torch.bfloat16).cuda()
    aux = torch.full((M, N), 0x7777, dtype=torch.int16, device="cuda").view(torch.bfloat16) \
        if act == fp8.ACT_GELU else h
    v32 = R.gemm(0, Av, afmt, 1, Bv, 0, out_dtype=fp8.OUT_F32, act=act, aux=aux, **kw)
    vb = R.gemm(0, Av, afmt, 1, Bv, 0, out_dtype=fp8.OUT_BF16, act=act,
                aux=h if act == fp8.ACT_DGELU else None, **kw)
    torch.cuda.synchronize()
    vmax = float(v32.abs().max())
    fmax = 448.0 if out_fmt == 0 else 57344.0
    s_out = float(np.float32(fmax / (0.5 * vmax)))  # some values saturate
    R.set_state(2, [0.5 * vmax] * 16, s_out, out_fmt)
    aux2 = torch.full((M, N), 0x1234, dtype=torch.int16, device="cuda").view(torch.bfloat16) \
        if act == fp8.ACT_GELU else h
    q = R.gemm(0, Av, afmt, 1, Bv, 0, out_dtype=2 + out_fmt, amax_out_id=2, act=act, aux=aux2, **kw)
    torch.cuda.synchronize()
    R.check_device_error()
    st2, _ = R.get_state(2)
    R.close()
    return dict(A=A, B=B, afmt=afmt, y32=y32.cpu().numpy(), v32=v32.cpu().numpy(), vb=to_host_u16(vb),
                q=to_host_u8(q), st=st2, s_out=s_out, h=None if h is None else to_host_u16(h),
                aux=None if act != fp8.ACT_GELU else (to_host_u16(aux), to_host_u16(aux2)),
                factor=np.float32(64.0) * np.float32(256.0))


def _check(fp8, r, act, out_fmt, rows):
    # bf16 output: RN of the same kernel's fp32 value
    assert np.array_equal(r["vb"], _bf16_rn(r["v32"])), "bf16 output is not RN(fp32 output)"
    # aux: bf16 of the kernel's plain product, from both launches that wrote it
    if act == fp8.ACT_GELU:
        want = _bf16_rn(r["y32"])
        assert np.array_equal(r["aux"][0], want) and np.array_equal(r["aux"][1], want), "aux != bf16(y)"
    # FP8 output and the output tensor's record: the oracle's epilogue cast of v
    oq, ns, nu, am = oracle.cast_f32(r["v32"], r["s_out"], out_fmt)
    bad = np.flatnonzero(r["q"].ravel() != oq.ravel())
    assert bad.size == 0, f"{bad.size} FP8 codes differ from the oracle's cast of v, first {bad[:4]}"
    st = r["st"]
    assert f32_bits(st["amax_pending"]) == f32_bits(am)
    assert st["n_saturated"] == ns and st["n_underflow"] == nu and ns > 0
    assert f32_bits(st["cast_scale"]) == f32_bits(np.float32(r["s_out"]))
    assert f32_bits(st["cast_scale_inv"]) == f32_bits(oracle.reciprocal(r["s_out"]))
    assert st["dtype"] == out_fmt and st["recorded"] == 1
    # the fp32 value against the oracle's fp64 chain, on the sampled rows
    f = r["factor"]
    acc, absacc, _ = oracle.gemm(r["A"], r["afmt"], r["B"], 0, f, rows=rows, want_bf16=False)
    y64 = acc * float(f)
    bound_y = 1e-6 * absacc * float(f)
    if act == fp8.ACT_GELU:
        v64 = oracle.gelu(y64)
        bound = _act_bound(y64, bound_y, act)
    else:
        hv = oracle.bf16_to_f32(r["h"][rows]).astype(np.float64)
        v64 = y64 * oracle.dgelu(hv)
        bound = _act_bound(y64, bound_y, act, hv)
    err = np.abs(r["v32"][rows].astype(np.float64) - v64)
    assert np.all(err <= bound), f"fp32 values beyond the bound: worst err/bound {np.max(err / bound):.3g}"


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("out_fmt", [0, 1])
def test_gelu_epilogue(gpu_lib, shape, out_fmt):
    M, N, K = shape
    r = _run(gpu_lib, M, N, K, gpu_lib.ACT_GELU, out_fmt, seed=M + 3 * N + 7 * K + out_fmt)
    _check(gpu_lib, r, gpu_lib.ACT_GELU, out_fmt, np.arange(0, M, max(1, M // 128)))


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("out_fmt", [1, 0])
def test_dgelu_epilogue(gpu_lib, shape, out_fmt):
    """FC2's dgrad: A = dY codes (E5M2), B = W codes read MN-major, as in the
    step."""
    M, N, K = shape
    r = _run(gpu_lib, M, N, K, gpu_lib.ACT_DGELU, out_fmt, seed=5 * M + N + K + out_fmt, b_major=1)
    _check(gpu_lib, r, gpu_lib.ACT_DGELU, out_fmt, np.arange(0, M, max(1, M // 128)))


def test_act_argument_checks(gpu_lib):
    fp8 = gpu_lib
    R = fp8.Recipe(3)
    A = torch.zeros((16, 32), dtype=torch.uint8, device="cuda")
    aux = torch.zeros((16, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp8.Fp8Error):  # GELU' needs the pre-activation
        R.gemm(0, A, 0, 1, A, 0, act=fp8.ACT_DGELU)
    with pytest.raises(fp8.Fp8Error):  # aux without an activation
        R.gemm(0, A, 0, 1, A, 0, aux=aux)
    with pytest.raises(fp8.Fp8Error):  # unknown activation
        R.gemm(0, A, 0, 1, A, 0, act=7)
    B = torch.zeros((12, 32), dtype=torch.uint8, device="cuda")
    aux12 = torch.zeros((16, 12), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp8.Fp8Error):  # N % 8 != 0: the aux rows are not whole 16-byte pieces
        R.gemm(0, A, 0, 1, B, 0, act=fp8.ACT_GELU, aux=aux12)
    R.close()
