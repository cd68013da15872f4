"""MX block scaling on the GPU against the oracle ("FP8 and low-precision
formats", format overview: per-block scale factors, MXFP8).

* fp8_mx_quantize: codes of x and of x^T and their E8M0 block scales, bit for
  bit against the oracle (the scales unpacked from the atom layout the C header
  documents; padding bytes must be 0).
* fp8_mx_gemm: every output (small shapes) or sampled rows and columns (large
  shapes) within mx_rel(K) * sum|a*b| of the oracle's fp64 sum for fp32
  outputs, and the bf16 rounding of a value inside that bound for bf16 outputs,
  1 ulp where the bound is tight.  Operands are quantised by the oracle on the
  host, so no oracle input comes from the GPU.

The tolerance comes from the arithmetic.  The tensor cores add each 32-element
block's scaled sum into an fp32 partial in TMEM; take every such add to be off
by up to one fp32 ulp of the running sum (2^-23 of its magnitude, which is at
most sum|a*b|).  The kernel starts a fresh partial every 64 blocks (K = 2048)
and adds the partials in round-to-nearest fp32 (2^-24 each), so
    |D - exact| <= (min(64, ceil(K/32)) * 2^-23 + ceil(K/2048) * 2^-24) * sum|a*b|,
about 7.6e-6 * sum|a*b| once K >= 2048.  (The per-tensor GEMM's 1e-6 does not
carry over: with block scales that differ by up to 2^48 along K, measured
errors reached 2.2e-6 * sum|a*b| at K = 4096 -- inside this bound -- and
promoting every block instead of every 64 left the typical error near
3e-7 while cutting throughput by a third.)
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_mixed_precision_history_gb300 import synthetic
from gpu_util import check_mx_gemm_sample, mx_atoms_from_plain, mx_plain_from_atoms, to_host_u8

pytestmark = pytest.mark.gpu

E4M3, E5M2 = oracle.E4M3, oracle.E5M2


def mx_rel(K):
    """Error bound of the MX GEMM as a fraction of sum|a*b| (module docstring)."""
    return min(64, -(-K // 32)) * 2.0 ** -23 + -(-K // 2048) * 2.0 ** -24


def _quantize_and_check(fp8, x, fmt, transpose):
    rows, cols = x.shape
    xb = synthetic.bits(x)
    R = fp8.Recipe(1)
    out = R.mx_quantize(x.cuda(), fmt, transpose=transpose)
    torch.cuda.synchronize()
    R.check_device_error()
    oq, osc = oracle.mx_quantize(xb, fmt)
    q = to_host_u8(out[0])
    bad = q != oq
    assert not bad.any(), f"{int(bad.sum())} codes differ; first at {np.argwhere(bad)[0]}"
    sc = mx_plain_from_atoms(to_host_u8(out[1]), rows, cols)
    bad = sc != osc
    assert not bad.any(), f"{int(bad.sum())} block scales differ; first at {np.argwhere(bad)[0]}"
    if transpose:
        oqt, osct = oracle.mx_quantize(np.ascontiguousarray(xb.T), fmt)
        qt = to_host_u8(out[2])
        bad = qt != oqt
        assert not bad.any(), f"{int(bad.sum())} transposed codes differ; first at {np.argwhere(bad)[0]}"
        sct = mx_plain_from_atoms(to_host_u8(out[3]), cols, rows)
        bad = sct != osct
        assert not bad.any(), f"{int(bad.sum())} transposed block scales differ"
    R.close()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("shape", [(128, 128), (304, 1008), (16, 48), (1024, 4096), (4096, 16384)])
def test_mx_quantize_matches_oracle(gpu_lib, fmt, shape):
    x = synthetic.block_varied(shape, 100 + shape[0] + shape[1] + fmt)
    _quantize_and_check(gpu_lib, x, fmt, transpose=True)


@pytest.mark.parametrize("shape", [(300, 1008), (1, 16), (130, 144)])
def test_mx_quantize_without_transpose_ragged_rows(gpu_lib, shape):
    x = synthetic.block_varied(shape, 7 + shape[0])
    _quantize_and_check(gpu_lib, x, E4M3, transpose=False)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_mx_quantize_edge_blocks(gpu_lib, fmt):
    """Blocks of zeros, of bf16 subnormals, near the largest bf16, and with
    amax exactly on / just above 1.75 * 2^e (the exponent's boundary)."""
    rows, cols = 32, 256
    rng = np.random.default_rng(4)
    v = (rng.standard_normal((rows, cols)) * 0.25).astype(np.float32)
    v[0, 0:32] = 0.0
    v[1, 32:64] = np.float32(2.0 ** -130) * rng.integers(-100, 100, 32)  # subnormal bf16 values
    v[2, 64:96] *= np.float32(2.0 ** 126)
    v[2, 70] = np.float32(1.9921875 * 2.0 ** 127)                        # largest bf16
    for j, e in enumerate(range(-20, 20, 5)):
        v[3 + j, 96:128] *= np.float32(2.0 ** e)
        v[3 + j, 100] = np.float32(1.75 * 2.0 ** e)
        v[3 + j, 128:160] *= np.float32(2.0 ** e)
        v[3 + j, 130] = np.float32(-1.7578125 * 2.0 ** e)
    v[20, :] = -0.0
    bits = (v.view(np.uint32) >> 16).astype(np.uint16)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    _quantize_and_check(gpu_lib, x, fmt, transpose=True)


def _operand(shape, fmt, seed, span=24, positive=False):
    x = synthetic.block_varied(shape, seed, span=span)
    if positive:
        x = x.abs()
    q, sc = oracle.mx_quantize(synthetic.bits(x), fmt)
    return q, sc


def _run_gemm(fp8, A, afmt, sa, B, bfmt, sb, M, N, K):
    R = fp8.Recipe(1)
    Ad = torch.from_numpy(A).cuda()
    Bd = torch.from_numpy(B).cuda()
    sad = torch.from_numpy(mx_atoms_from_plain(sa, M, K)).cuda()
    sbd = torch.from_numpy(mx_atoms_from_plain(sb, N, K)).cuda()
    D32 = R.mx_gemm(Ad, afmt, sad, Bd, bfmt, sbd, out_dtype=fp8.OUT_F32)
    Db = R.mx_gemm(Ad, afmt, sad, Bd, bfmt, sbd, out_dtype=fp8.OUT_BF16)
    torch.cuda.synchronize()
    R.check_device_error()
    R.close()
    return D32, Db


@pytest.mark.parametrize("fmts", [(E4M3, E4M3), (E5M2, E4M3), (E5M2, E5M2)])
@pytest.mark.parametrize("shape", [(256, 512, 512), (129, 264, 144), (300, 1000, 208), (64, 512, 32),
                                   (1024, 1024, 4096), (4096, 4096, 2336)])
def test_mx_gemm_matches_oracle(gpu_lib, fmts, shape):
    M, N, K = shape
    afmt, bfmt = fmts
    A, sa = _operand((M, K), afmt, M + K + afmt)
    B, sb = _operand((N, K), bfmt, N + K + 10 * bfmt + 1)
    D32, Db = _run_gemm(gpu_lib, A, afmt, sa, B, bfmt, sb, M, N, K)
    if M * N * K <= 300 * 1000 * 208:
        check_mx_gemm_sample(D32, Db, A, afmt, sa, B, bfmt, sb, rows=np.arange(M), rel=mx_rel(K))
    else:
        rng = np.random.default_rng(M + N)
        check_mx_gemm_sample(D32, Db, A, afmt, sa, B, bfmt, sb, rows=np.sort(rng.choice(M, 64, replace=False)),
                             cols=np.sort(rng.choice(N, 64, replace=False)), rel=mx_rel(K))


def test_mx_gemm_long_k_same_sign(gpu_lib):
    """K = 16384 with every product positive and comparable: the sum most
    exposed to accumulation error (eight promoted partials)."""
    M, N, K = 128, 256, 16384
    A, sa = _operand((M, K), E4M3, 5, span=1, positive=True)
    B, sb = _operand((N, K), E4M3, 6, span=1, positive=True)
    D32, Db = _run_gemm(gpu_lib, A, E4M3, sa, B, E4M3, sb, M, N, K)
    check_mx_gemm_sample(D32, Db, A, E4M3, sa, B, E4M3, sb, rows=np.arange(0, M, 3), rel=mx_rel(K))


def test_mx_gemm_full_size_fc2(gpu_lib):
    """The FC2 forward shape, M=8192 N=4096 K=16384: sampled rows and columns."""
    M, N, K = 8192, 4096, 16384
    A, sa = _operand((M, K), E4M3, 21)
    B, sb = _operand((N, K), E4M3, 22)
    D32, Db = _run_gemm(gpu_lib, A, E4M3, sa, B, E4M3, sb, M, N, K)
    rng = np.random.default_rng(3)
    check_mx_gemm_sample(D32, Db, A, E4M3, sa, B, E4M3, sb, rows=np.sort(rng.choice(M, 24, replace=False)),
                         cols=np.sort(rng.choice(N, 12, replace=False)), rel=mx_rel(K))


def test_mx_linear_layer_chain(gpu_lib):
    """Forward, dgrad and wgrad of one linear layer through the GPU quantiser
    (X, W in E4M3, dY in E5M2, each with its transposed copy) and the MX GEMM;
    the oracle quantises the same bf16 tensors itself and runs its own GEMMs."""
    fp8 = gpu_lib
    T, fin, fout = 256, 384, 512
    x = synthetic.normal((T, fin), 1.0, 31)
    w = synthetic.normal((fout, fin), 0.02, 32)
    dy = synthetic.grad_like((T, fout), 33)
    R = fp8.Recipe(1)
    qx, sx, qxt, sxt = R.mx_quantize(x.cuda(), E4M3, transpose=True)
    qw, sw, qwt, swt = R.mx_quantize(w.cuda(), E4M3, transpose=True)
    qd, sd, qdt, sdt = R.mx_quantize(dy.cuda(), E5M2, transpose=True)
    y = R.mx_gemm(qx, E4M3, sx, qw, E4M3, sw, out_dtype=fp8.OUT_F32)
    dx = R.mx_gemm(qd, E5M2, sd, qwt, E4M3, swt, out_dtype=fp8.OUT_F32)
    dw = R.mx_gemm(qdt, E5M2, sdt, qxt, E4M3, sxt, out_dtype=fp8.OUT_F32)
    torch.cuda.synchronize()
    R.check_device_error()
    R.close()
    ox, osx = oracle.mx_quantize(synthetic.bits(x), E4M3)
    ow, osw = oracle.mx_quantize(synthetic.bits(w), E4M3)
    od, osd = oracle.mx_quantize(synthetic.bits(dy), E5M2)
    owt, oswt = oracle.mx_quantize(np.ascontiguousarray(synthetic.bits(w).T), E4M3)
    oxt, osxt = oracle.mx_quantize(np.ascontiguousarray(synthetic.bits(x).T), E4M3)
    odt, osdt = oracle.mx_quantize(np.ascontiguousarray(synthetic.bits(dy).T), E5M2)
    check_mx_gemm_sample(y, None, ox, E4M3, osx, ow, E4M3, osw, rows=np.arange(T), rel=mx_rel(fin))
    check_mx_gemm_sample(dx, None, od, E5M2, osd, owt, E4M3, oswt, rows=np.arange(T), rel=mx_rel(fout))
    check_mx_gemm_sample(dw, None, odt, E5M2, osdt, oxt, E4M3, osxt, rows=np.arange(fout), rel=mx_rel(T))


def test_mx_argument_checks(gpu_lib):
    fp8 = gpu_lib
    R = fp8.Recipe(1)
    x = torch.zeros((20, 48), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp8.Fp8Error):
        R.mx_quantize(x, E4M3, transpose=True)  # rows % 16 != 0 with a transposed copy
    x = torch.zeros((16, 40), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp8.Fp8Error):
        R.mx_quantize(x, E4M3)  # cols % 16 != 0
    A = torch.zeros((16, 32), dtype=torch.uint8, device="cuda")
    s = torch.zeros(512, dtype=torch.uint8, device="cuda")
    with pytest.raises(fp8.Fp8Error):
        R.mx_gemm(A, E4M3, s, A, E4M3, s, out_dtype=fp8.OUT_E4M3)  # FP8 outputs are per-tensor only
    R.close()
