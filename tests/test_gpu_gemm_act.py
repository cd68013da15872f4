"""GEMM with the MLP's activation fused into the epilogue (fp8_gemm_act).

"4.2 Hopper I -- Transformer Engine / FP8", S4.2.4: the FP32 result is
multiplied by 1/scale "or composed with the next stage's scale"; S4.2.6's
te.TransformerLayer puts an activation between FC1 and FC2 (GELU, tanh form:
the reading taken).  FC1's forward stores gelu(y) -- as FC2's E4M3 operand --
and bf16(gelu'(y)) for the backward; FC2's dgrad stores y * gelu' (the saved
derivative) -- as FC1's E5M2 output gradient.

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
* the aux output bf16(gelu'(y)) is the same from every launch and lies within
  one bf16 spacing (plus the propagated bounds) of the oracle's gelu'(y).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import bf16_spacing, f32_bits, to_host_u16, to_host_u8
from test_gpu_gemm import _device_operand, _tensor_codes

pytestmark = pytest.mark.gpu

SHAPES = [(256, 512, 512), (129, 264, 144), (300, 1000, 208), (64, 512, 32), (1024, 1024, 4096),
          (384, 2048, 2048), (200, 136, 4112)]


def _bf16_rn(v32):
    return torch.from_numpy(np.ascontiguousarray(v32, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


C_GELU, A_GELU = np.sqrt(2.0 / np.pi), 0.044715


def _dgelu_eval_bound(x):
    """fp32 evaluation error of gelu'(x) in the sigmoid form s = 1/(1 + e^-z),
    z = 2c (x + a x^3), gelu' = s + 2x s (1-s) c (1 + 3a x^2): the fast
    exponential (relative error within (2 + 1.5|z|) ulp, z itself off by three
    roundings) and the approximate reciprocal leave s within 2^-20 (2 + 2|z|)
    of its relative value and the product term within 2^-19 (1 + |z|)."""
    z = 2 * C_GELU * (x + A_GELU * x ** 3)
    sg = 1.0 / (1.0 + np.exp(-np.clip(z, -80, 80)))
    term = np.abs(2 * x * sg * (1 - sg) * C_GELU * (1 + 3 * A_GELU * x * x))
    return 2.0 ** -19 * (1 + np.abs(z)) * (sg + term)


def _act_bound(y64, bound_y, act, g=None):
    """|v_gpu - v_oracle| for v = gelu(y), or y * g with g the given bf16
    derivative (exactly decoded).
    gelu: the GEMM leaves |y32 - y64| <= bound_y and |gelu'| <= 1.2, so gelu
    moves it by at most 1.2 bound_y; the fp32 evaluation through
    s = 1/(1 + e^-z) (fast exponential within (2 + 1.5|z|) ulp, z off by three
    roundings, approximate reciprocal) leaves gelu = x s within
    2^-20 (2 + 2|z|) |gelu|.
    y * g: |g| bound_y plus two roundings (y * factor, then * g)."""
    if act == 1:
        z = np.abs(2 * C_GELU * (y64 + A_GELU * y64 ** 3))
        return 1.2 * bound_y + 2.0 ** -20 * (2 + 2 * z) * np.abs(oracle.gelu(y64))
    return np.abs(g) * bound_y + 2.0 ** -23 * np.abs(y64 * g)


def _aux_bound(y64, bound_y):
    """|bf16(gelu'_gpu(y32)) - gelu'(y64)|: gelu'' is within 0.8 in magnitude,
    so the GEMM error moves gelu' by at most 0.8 bound_y; then the fp32
    evaluation and one bf16 rounding (at most one bf16 spacing with the
    evaluation error near a rounding boundary)."""
    dg = oracle.dgelu(y64)
    return 0.8 * bound_y + _dgelu_eval_bound(y64) + bf16_spacing(np.abs(dg) + 0.8 * bound_y)


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
    if act == fp8.ACT_DGELU:  # the forward's saved derivative: bf16 gelu' of values around the bend
        g = oracle.f64_to_bf16(oracle.dgelu(rng.standard_normal((M, N)) * 1.5))
        h = torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).cuda()
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
    # aux: the same bf16 derivative from both launches that wrote it
    if act == fp8.ACT_GELU:
        assert np.array_equal(r["aux"][0], r["aux"][1]), "the launches wrote different aux values"
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
        aux = oracle.bf16_to_f32(r["aux"][0][rows]).astype(np.float64)
        aerr = np.abs(aux - oracle.dgelu(y64))
        abound = _aux_bound(y64, bound_y)
        assert np.all(aerr <= abound), f"aux beyond the bound: worst err/bound {np.max(aerr / abound):.3g}"
    else:
        gv = oracle.bf16_to_f32(r["h"][rows]).astype(np.float64)
        v64 = y64 * gv
        bound = _act_bound(y64, bound_y, act, gv)
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
