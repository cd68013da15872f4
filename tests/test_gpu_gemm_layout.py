"""GEMM with MN-major operands (fp8_gemm_layout) against the oracle.

"4.2 Hopper I -- Transformer Engine / FP8", S4.2.4: the three GEMMs of a linear
layer -- forward Y = X W^T, dgrad dX = dY W, wgrad dW = dY^T X -- on FP8 codes
with FP32 accumulation and 1/scale dequantisation.  On these tensor cores the
backward GEMMs read the forward casts' codes directly: W [out, in] is dgrad's
B operand stored MN-major; dY [T, out] and X [T, in] are wgrad's A and B stored
MN-major.  The oracle is given the same codes as [M, K] and [N, K] matrices (a
host-side transpose of the stored array), and every output is held to the
bounds of the K-major tests."""
import numpy as np
import pytest
import torch

import oracle
from fp8_mixed_precision_history_gb300 import synthetic
from gpu_util import check_gemm_sample, fp32_mma_rel, to_host_u8
from test_gpu_gemm import _finite_codes, _full_check, _tensor_codes

pytestmark = pytest.mark.gpu

LAYOUTS = [(0, 1), (1, 0), (1, 1)]  # (a_major, b_major); 1 = MN-major
SHAPES = [(256, 512, 512), (1, 8, 16), (16, 16, 16), (129, 257, 144), (200, 300, 208),
          (128, 256, 128), (384, 1024, 2048), (272, 528, 4112), (64, 600, 32), (272, 528, 112)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("combo", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_layout_tensor_codes(gpu_lib, shape, layout, combo):
    """Operands distributed like the pages' cast tensors: the 1e-6 bound.
    Shapes span several tiles with ragged M, N and K tails."""
    M, N, K = shape
    afmt, bfmt = combo
    rng = np.random.default_rng(M * 1000003 + N * 1009 + K + 17 * afmt + 5 * bfmt + 31 * layout[0] + 7 * layout[1])
    A = _tensor_codes(rng, (M, K), afmt)
    B = _tensor_codes(rng, (N, K), bfmt)
    _full_check(gpu_lib, A, afmt, B, bfmt, sa=1.0 / 64, sb=1.0 / 256, a_major=layout[0], b_major=layout[1])


@pytest.mark.parametrize("shape", [(129, 257, 144), (384, 1024, 2048), (272, 528, 4112)])
@pytest.mark.parametrize("layout", LAYOUTS)
def test_layout_random_codes(gpu_lib, shape, layout):
    """Uniformly random finite codes against the bound of the kernel's FP32
    accumulation (fp32_mma_rel): a misplaced element of either operand shows."""
    M, N, K = shape
    rng = np.random.default_rng(M + N + K + 3 * layout[0] + layout[1])
    A = _finite_codes(rng, (M, K), 1, max_code=0x5C)
    B = _finite_codes(rng, (N, K), 0, max_code=0x70)
    _full_check(gpu_lib, A, 1, B, 0, rel=fp32_mma_rel(K), a_major=layout[0], b_major=layout[1])


@pytest.mark.parametrize("layout", LAYOUTS)
def test_layout_strided_views(gpu_lib, layout):
    """MN-major views into wider buffers (row stride > M or N); ldd > N."""
    rng = np.random.default_rng(5 + layout[0])
    M, N, K = 300, 264, 160
    A = _finite_codes(rng, (M, K), 0, 0x68)
    B = _finite_codes(rng, (N, K), 1, 0x50)
    lda = 320 if layout[0] else 208
    ldb = 288 if layout[1] else 176
    _full_check(gpu_lib, A, 0, B, 1, lda=lda, ldb=ldb, ldd=296, a_major=layout[0], b_major=layout[1])


def test_layout_all_positive_k16384(gpu_lib):
    """All-positive operands at K = 16384, both MN-major (the wgrad layout)."""
    rng = np.random.default_rng(12)
    M, N, K = 128, 256, 16384
    A = rng.integers(0x30, 0x48, (M, K)).astype(np.uint8)
    B = rng.integers(0x30, 0x48, (N, K)).astype(np.uint8)
    _full_check(gpu_lib, A, 0, B, 0, sa=1.0, sb=1.0, a_major=1, b_major=1)


@pytest.mark.parametrize("out", [2, 3])
def test_layout_fp8_output(gpu_lib, out):
    """FP8-output epilogue on MN-major operands: the codes equal the saturating
    cast of the same call's fp32 output, which meets the oracle's bound."""
    fp8 = gpu_lib
    M, N, K = 304, 528, 272  # MN-major row strides are multiples of 16 bytes; ragged tiles
    rng = np.random.default_rng(40 + out)
    afmt, bfmt = (1, 0)
    A = _tensor_codes(rng, (M, K), afmt)
    B = _tensor_codes(rng, (N, K), bfmt)
    R = fp8.Recipe(3)
    R.set_state(0, [1.0] * 16, 1.0 / 64, afmt)
    R.set_state(1, [1.0] * 16, 1.0 / 256, bfmt)
    At = torch.from_numpy(np.ascontiguousarray(A.T)).cuda()
    Bt = torch.from_numpy(np.ascontiguousarray(B.T)).cuda()
    kw = dict(a_major=1, b_major=1)
    y32 = R.gemm(0, At, afmt, 1, Bt, bfmt, out_dtype=fp8.OUT_F32, **kw)
    torch.cuda.synchronize()
    factor = np.float32(R.get_state(0)[0]["cast_scale_inv"]) * np.float32(R.get_state(1)[0]["cast_scale_inv"])
    check_gemm_sample(y32, None, A, afmt, B, bfmt, factor, np.arange(M))
    s_out = float(np.float32((448.0 if out == 2 else 57344.0) / (0.5 * float(y32.abs().max()))))
    R.set_state(2, [0.5] * 16, s_out, out - 2)
    D8 = R.gemm(0, At, afmt, 1, Bt, bfmt, out_dtype=out, amax_out_id=2, **kw)
    torch.cuda.synchronize()
    R.check_device_error()
    lim = 448.0 if out == 2 else 57344.0
    want = (y32 * np.float32(s_out)).clamp(-lim, lim).to(torch.float8_e4m3fn if out == 2 else torch.float8_e5m2)
    assert torch.equal(D8.view(torch.uint8), want.view(torch.uint8))
    R.close()


def test_layout_matches_k_major_bits(gpu_lib):
    """The same product read through either layout: identical fp32 outputs on
    data whose every partial sum is exact (small integers), so any difference
    would be a misread element, not rounding."""
    fp8 = gpu_lib
    rng = np.random.default_rng(9)
    M, N, K = 384, 768, 1040
    # E4M3 codes of the integers -4..4 (exact products and sums in fp32)
    vals = rng.integers(-4, 5, (M, K)).astype(np.float32)
    A = oracle.encode(vals, oracle.E4M3)
    B = oracle.encode(rng.integers(-4, 5, (N, K)).astype(np.float32), oracle.E4M3)
    R = fp8.Recipe(2)
    R.set_state(0, [1.0] * 16, 1.0, 0)
    R.set_state(1, [1.0] * 16, 1.0, 0)
    exact = vals.astype(np.float64) @ oracle.decode(B, oracle.E4M3).astype(np.float64).T
    for a_major in (0, 1):
        for b_major in (0, 1):
            Av = torch.from_numpy(A if a_major == 0 else np.ascontiguousarray(A.T)).cuda()
            Bv = torch.from_numpy(B if b_major == 0 else np.ascontiguousarray(B.T)).cuda()
            y = R.gemm(0, Av, 0, 1, Bv, 0, out_dtype=fp8.OUT_F32, a_major=a_major, b_major=b_major)
            torch.cuda.synchronize()
            assert np.array_equal(y.cpu().numpy().astype(np.float64), exact), (a_major, b_major)
    R.close()


def test_layout_argument_checks(gpu_lib):
    fp8 = gpu_lib
    R = fp8.Recipe(2)
    A = torch.zeros((64, 48), dtype=torch.uint8, device="cuda")  # MN-major: K = 64, M = 48
    B = torch.zeros((64, 32), dtype=torch.uint8, device="cuda")
    D = torch.zeros((48, 32), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp8.Fp8Error):  # unknown layout
        fp8.fp8_gemm_layout(R.handle, 0, A, 0, 2, 48, 1, B, 0, 1, 32, 48, 32, 64, D, 0, 32)
    with pytest.raises(fp8.Fp8Error):  # MN-major A: lda < M
        fp8.fp8_gemm_layout(R.handle, 0, A, 0, 1, 32, 1, B, 0, 1, 32, 48, 32, 64, D, 0, 32)
    with pytest.raises(fp8.Fp8Error):  # MN-major B: ldb not a multiple of 16
        fp8.fp8_gemm_layout(R.handle, 0, A, 0, 1, 48, 1, B, 0, 1, 40, 48, 32, 64, D, 0, 32)
    fp8.fp8_gemm_layout(R.handle, 0, A, 0, 1, 48, 1, B, 0, 1, 32, 48, 32, 64, D, 0, 32)
    torch.cuda.synchronize()
    R.check_device_error()
    R.close()


@pytest.mark.parametrize("layer", [0, 1, 2, 3])
def test_te_layer_backward_without_transposes(gpu_lib, layer):
    """The transformer layer's backward GEMMs at full size (8192 tokens) on the
    forward casts' codes -- no transposed copies -- in the launch configuration
    of the step: sampled rows and columns against the oracle."""
    fp8 = gpu_lib
    T = 8192
    _, fin, fout = synthetic.TE_LAYERS[layer]
    x = synthetic.normal((T, fin), 1.0, synthetic.seed_for(3, layer, "x"), device="cuda")
    w = synthetic.normal((fout, fin), 0.02, synthetic.seed_for(3, layer, "w"), device="cuda")
    dy = synthetic.grad_like((T, fout), synthetic.seed_for(4, layer, "dy"), device="cuda")
    R = fp8.Recipe(3)
    xq = R.quantize(0, x, fp8.E4M3, fp8.CURRENT)
    wq = R.quantize(1, w, fp8.E4M3, fp8.CURRENT)
    dq = R.quantize(2, dy, fp8.E5M2, fp8.CURRENT)
    sinv = [np.float32(R.get_state(t)[0]["cast_scale_inv"]) for t in range(3)]
    hx, hw, hd = to_host_u8(xq), to_host_u8(wq), to_host_u8(dq)
    rng = np.random.default_rng(200 + layer)
    cases = [  # name, A, afmt, a_id, a_major, B, bfmt, b_id, b_major, host A [M,K], host B [N,K]
        ("dgrad", dq, 1, 2, 0, wq, 0, 1, 1, hd, np.ascontiguousarray(hw.T)),
        ("wgrad", dq, 1, 2, 1, xq, 0, 0, 1, np.ascontiguousarray(hd.T), np.ascontiguousarray(hx.T)),
    ]
    for name, A, afmt, aid, am, B, bfmt, bid, bm, hA, hB in cases:
        D32 = R.gemm(aid, A, afmt, bid, B, bfmt, out_dtype=fp8.OUT_F32, a_major=am, b_major=bm)
        Db = R.gemm(aid, A, afmt, bid, B, bfmt, a_major=am, b_major=bm)
        torch.cuda.synchronize()
        R.check_device_error()
        M, N = hA.shape[0], hB.shape[0]
        assert D32.shape == (M, N)
        rows = np.sort(rng.choice(M, 192, replace=False))
        cols = np.sort(rng.choice(N, 192, replace=False))
        worst = check_gemm_sample(D32, Db, hA, afmt, hB, bfmt, sinv[aid] * sinv[bid], rows, cols)
        assert worst <= 1, name
        del D32, Db
    R.close()
