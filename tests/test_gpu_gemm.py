"""GPU parity of the tcgen05 FP8 GEMM against the oracle.

Bound ("4.2 Hopper I -- Transformer Engine / FP8", S4.2.4: FP8 inputs, FP32
accumulation, x 1/scale): every fp32 output within 1e-6 * sum_k |a*b| * factor
of the oracle's fp64 result for operands distributed like the pages' tensors
(for uniformly random codes, the bound of the FP32 accumulation with its
promotion every 2048 of K, gpu_util.fp32_mma_rel); every bf16 output the rounding of a value inside that bound, and within
1 ulp of the oracle's bf16 wherever the bound is below half a bf16 spacing; bf16
output == RN(fp32 output) bit for bit; a fused output amax equal to max|D| of
the stored values."""
import numpy as np
import pytest
import torch

import oracle
from fp8_mixed_precision_history_gb300 import synthetic
from gpu_util import bf16_ord, check_gemm_sample, f32_bits, fp32_mma_rel, to_host_u16, to_host_u8

pytestmark = pytest.mark.gpu

COMBOS = [(0, 0), (1, 0), (0, 1), (1, 1)]


def _finite_codes(rng, shape, fmt, max_code=None):
    c = rng.integers(0, 256, shape).astype(np.uint8)
    top = (0x7E if fmt == 0 else 0x7B) if max_code is None else max_code
    mag = c & 0x7F
    mag = np.where(mag > top, mag % (top + 1), mag).astype(np.uint8)
    return (c & 0x80) | mag


def _recipe_with_scales(fp8, sa, sb, fa, fb):
    R = fp8.Recipe(3)
    R.set_state(0, [1.0] * 16, sa, fa)
    R.set_state(1, [1.0] * 16, sb, fb)
    return R


def _device_operand(codes, major, ld):
    """Host codes [rows, K] stored on the GPU K-major ([rows, K], row stride
    ld >= K) or MN-major ([K, rows], row stride ld >= rows); returns the view."""
    stored = codes if major == 0 else np.ascontiguousarray(codes.T)
    r, c = stored.shape
    ld = ld or -(-c // 16) * 16  # row strides are multiples of 16 bytes
    d = torch.zeros((r, ld), dtype=torch.uint8, device="cuda")
    d[:, :c] = torch.from_numpy(stored).cuda()
    return d[:, :c]


def _full_check(fp8, A, afmt, B, bfmt, sa=2.0, sb=0.5, lda=None, ldb=None, ldd=None, rel=1e-6,
                a_major=0, b_major=0):
    """A [M, K], B [N, K] host codes; on the GPU either may be stored MN-major."""
    M, K = A.shape
    N = B.shape[0]
    R = _recipe_with_scales(fp8, sa, sb, afmt, bfmt)
    Av = _device_operand(A, a_major, lda)
    Bv = _device_operand(B, b_major, ldb)
    D32 = torch.full((M, ldd or N), -7.0, dtype=torch.float32, device="cuda")
    Db = torch.full((M, ldd or N), 12345, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    kw = dict(a_major=a_major, b_major=b_major)
    R.gemm(0, Av, afmt, 1, Bv, bfmt, out_dtype=fp8.OUT_F32, out=D32[:, :N], **kw)
    R.gemm(0, Av, afmt, 1, Bv, bfmt, out_dtype=fp8.OUT_BF16, out=Db[:, :N], amax_out_id=2, **kw)
    torch.cuda.synchronize()
    R.check_device_error()
    if ldd and ldd > N:  # padding columns untouched
        assert torch.all(D32[:, N:] == -7.0)
        assert torch.all(Db[:, N:].view(torch.int16) == 12345)
    st0, _ = R.get_state(0)
    st1, _ = R.get_state(1)
    factor = np.float32(st0["cast_scale_inv"]) * np.float32(st1["cast_scale_inv"])
    assert f32_bits(st0["cast_scale_inv"]) == f32_bits(oracle.reciprocal(sa))
    rows = np.arange(M)
    worst = check_gemm_sample(D32[:, :N], Db[:, :N], A, afmt, B, bfmt, factor, rows, rel=rel)
    # fused amax: exactly max|D| of what was stored, within 1 ulp of the oracle's
    st2, _ = R.get_state(2)
    gb = to_host_u16(Db[:, :N]).astype(np.uint32)
    mine = np.float32(np.max(np.abs((gb << 16).view(np.float32))))
    assert f32_bits(st2["amax_pending"]) == f32_bits(mine)
    _, _, ob = oracle.gemm(A, afmt, B, bfmt, factor)
    omax = np.max(bf16_ord(ob) * np.sign(bf16_ord(ob)))
    gmax = int(f32_bits(mine) >> 16)
    assert abs(gmax - int(omax)) <= 1
    R.close()
    return worst


# M > 128 runs the two-CTA kernel (256-byte K stages: with K <= 128 a K-major
# operand's second 128-byte box lies wholly past K and reads zeros), M <= 128
# the one-CTA kernel
SHAPES = [(256, 512, 512), (1, 8, 16), (1, 1, 16), (129, 257, 144), (200, 300, 208),
          (128, 256, 128), (384, 1024, 2048), (257, 513, 4112), (64, 600, 32), (256, 512, 16),
          (300, 264, 112)]


def _tensor_codes(rng, shape, fmt):
    """Codes of a cast tensor: N(0,1) activations/weights scaled so amax ~ FP8_MAX
    (E4M3), or signed log-uniform gradients on [1e-6, 1e-1] scaled likewise (E5M2)."""
    if fmt == 0:
        v = rng.standard_normal(shape) * (448.0 / 4.5)
    else:
        mag = np.exp(rng.uniform(np.log(1e-6), np.log(1e-1), shape)) * (57344.0 / 0.1)
        v = np.where(rng.random(shape) < 0.5, -mag, mag)
    return oracle.encode(v.astype(np.float32), fmt)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("combo", COMBOS)
def test_gemm_full_tensor_codes(gpu_lib, shape, combo):
    """Operands distributed like the pages' cast tensors: the 1e-6 bound."""
    M, N, K = shape
    afmt, bfmt = combo
    rng = np.random.default_rng(M * 1000003 + N * 1009 + K + 17 * afmt + 5 * bfmt)
    A = _tensor_codes(rng, (M, K), afmt)
    B = _tensor_codes(rng, (N, K), bfmt)
    _full_check(gpu_lib, A, afmt, B, bfmt, sa=1.0 / 64, sb=1.0 / 256)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("combo", COMBOS)
def test_gemm_full_random_codes(gpu_lib, shape, combo):
    """Uniformly random finite codes: products spread over the whole exponent
    range, so a few terms dominate each sum and fp32 accumulation rounds at
    their scale.  Checked against the bound of the kernel's FP32 accumulation
    (two roundings per K = 32 step inside a 2048-deep partial, partials
    promoted into round-to-nearest fp32), fp32_mma_rel(K)."""
    M, N, K = shape
    afmt, bfmt = combo
    rng = np.random.default_rng(M * 1000003 + N * 1009 + K + 17 * afmt + 5 * bfmt + 1)
    # keep products moderate so that fp32 output never overflows
    A = _finite_codes(rng, (M, K), afmt, max_code=0x70 if afmt == 0 else 0x5C)
    B = _finite_codes(rng, (N, K), bfmt, max_code=0x70 if bfmt == 0 else 0x5C)
    _full_check(gpu_lib, A, afmt, B, bfmt, rel=fp32_mma_rel(K))


@pytest.mark.parametrize("M", [128, 256])
@pytest.mark.parametrize("combo", COMBOS)
def test_gemm_random_codes_long_k(gpu_lib, M, combo):
    """K = 16384 (eight 2048-deep partials) on uniformly random codes, M = 128
    and 256: the accumulation bound stays that of a single partial, so a
    kernel that stopped promoting would fail it.  Both run the two-CTA kernel
    with the tile's partials split across pairs (a single 128- or 256-row
    tile meeting a long K); test_gpu_gemm_one runs them on the one-CTA kernel."""
    K = 16384
    afmt, bfmt = combo
    rng = np.random.default_rng(M + 41 * afmt + 7 * bfmt)
    A = _finite_codes(rng, (M, K), afmt, max_code=0x70 if afmt == 0 else 0x5C)
    B = _finite_codes(rng, (256, K), bfmt, max_code=0x70 if bfmt == 0 else 0x5C)
    _full_check(gpu_lib, A, afmt, B, bfmt, rel=fp32_mma_rel(K))


# Shapes whose last wave of 256 x 256 tiles the two-CTA kernel shares out by
# TMEM partial (2048 of K) across every CTA pair (76 on a GB300):
#   (512, 1024, 16384): 8 tiles of 8 partials on 64 pairs -- each tile an
#     owner and seven helpers;
#   (1280, 2560, 6144): 50 tiles of 3 partials on 76 pairs -- pairs holding a
#     helper piece and then an owner piece;
#   (4096, 5120, 4112): 320 tiles, four whole waves, then the last 16 tiles'
#     three partials (the last one 16 deep) split.
SPLIT_SHAPES = [((512, 1024, 16384), (0, 0)), ((1280, 2560, 6144), (1, 0)), ((4096, 5120, 4112), (0, 1))]


@pytest.mark.parametrize("shape,combo", SPLIT_SHAPES)
def test_gemm_split_tail(gpu_lib, shape, combo):
    """Sampled rows (every column) against the oracle within the accumulation
    bound, and the same bits from a second launch: a split tile's sum does
    not depend on the order in which its pieces finish."""
    fp8 = gpu_lib
    M, N, K = shape
    afmt, bfmt = combo
    rng = np.random.default_rng(M + N + K)
    A = _finite_codes(rng, (M, K), afmt, max_code=0x70 if afmt == 0 else 0x5C)
    B = _finite_codes(rng, (N, K), bfmt, max_code=0x70 if bfmt == 0 else 0x5C)
    R = _recipe_with_scales(fp8, 2.0, 0.5, afmt, bfmt)
    Av, Bv = _device_operand(A, 0, None), _device_operand(B, 0, None)
    D1 = R.gemm(0, Av, afmt, 1, Bv, bfmt, out_dtype=fp8.OUT_F32)
    D2 = R.gemm(0, Av, afmt, 1, Bv, bfmt, out_dtype=fp8.OUT_F32)
    Db = R.gemm(0, Av, afmt, 1, Bv, bfmt)
    torch.cuda.synchronize()
    R.check_device_error()
    assert torch.equal(D1.view(torch.int32), D2.view(torch.int32))
    factor = np.float32(0.5) * np.float32(2.0)
    rows = np.unique(np.concatenate([np.arange(0, M, max(1, M // 48)), [M - 1]]))
    check_gemm_sample(D1, Db, A, afmt, B, bfmt, factor, rows, rel=fp32_mma_rel(K))
    R.close()


def test_gemm_split_tail_graph_replay(gpu_lib):
    """A captured split-tile GEMM replayed on new operand values: every replay
    must wait for its own helpers' sums (the flags' epoch lives on the device,
    so a replay cannot match flags a previous launch left)."""
    fp8 = gpu_lib
    M, N, K = 512, 1024, 16384
    rng = np.random.default_rng(7)
    B = _finite_codes(rng, (N, K), 0, max_code=0x70)
    R = _recipe_with_scales(fp8, 2.0, 0.5, 0, 0)
    Bv = _device_operand(B, 0, None)
    A0 = _finite_codes(rng, (M, K), 0, max_code=0x70)
    Av = _device_operand(A0, 0, None)
    D = torch.empty((M, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        R.gemm(0, Av, 0, 1, Bv, 0, out_dtype=fp8.OUT_F32, out=D, stream=s)  # set-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        R.gemm(0, Av, 0, 1, Bv, 0, out_dtype=fp8.OUT_F32, out=D, stream=torch.cuda.current_stream())
    rows = np.arange(0, M, 16)
    for trial in range(3):
        A = _finite_codes(rng, (M, K), 0, max_code=0x70)
        Av.copy_(torch.from_numpy(A).cuda())
        g.replay()
        torch.cuda.synchronize()
        R.check_device_error()
        eager = R.gemm(0, Av, 0, 1, Bv, 0, out_dtype=fp8.OUT_F32)
        torch.cuda.synchronize()
        assert torch.equal(D.view(torch.int32), eager.view(torch.int32)), f"replay {trial} differs from a launch"
        check_gemm_sample(D, None, A, 0, B, 0, np.float32(1.0), rows, rel=fp32_mma_rel(K))
    R.close()


@pytest.mark.parametrize("n,ldd", [(270, 280), (264, 296), (520, 640)])
def test_gemm_strided_views(gpu_lib, n, ldd):
    """Views into wider buffers (lda, ldb > K; ldd > N): columns past N untouched.
    N = 264 and 520 take the TMA-store epilogue, N = 270 the direct stores."""
    rng = np.random.default_rng(3 + n)
    A = _finite_codes(rng, (300, 160), 0, 0x68)
    B = _finite_codes(rng, (n, 160), 1, 0x50)
    _full_check(gpu_lib, A, 0, B, 1, lda=208, ldb=176, ldd=ldd)


def test_gemm_single_linear_forward(gpu_lib):
    """Delayed-scaling FP8 linear forward: X [256,512], W [512,512] ~ N(0, 0.02)
    from seed 0, histories pre-filled with each tensor's amax, E4M3 casts."""
    fp8 = gpu_lib
    x, w = synthetic.single_linear(seed=0)
    R = fp8.Recipe(3)
    OR = oracle.DelayedRecipe(3)
    for tid, t in ((0, x), (1, w)):
        b = synthetic.bits(t)
        a = float(oracle.amax(b))
        s = float(oracle.scale_from_amax(a, 0))
        R.set_state(tid, [a] * 16, s, 0)
        OR.set_state(tid, [a] * 16, s, 0)
    xq = R.quantize(0, x.cuda(), 0)
    wq = R.quantize(1, w.cuda(), 0)
    y32 = R.gemm(0, xq, 0, 1, wq, 0, out_dtype=fp8.OUT_F32)
    yb = R.gemm(0, xq, 0, 1, wq, 0)
    oxq = OR.quantize(0, synthetic.bits(x), 0)
    owq = OR.quantize(1, synthetic.bits(w), 0)
    assert np.array_equal(to_host_u8(xq), oxq) and np.array_equal(to_host_u8(wq), owq)
    factor = np.float32(OR.t[0].cast_scale_inv) * np.float32(OR.t[1].cast_scale_inv)
    check_gemm_sample(y32, yb, oxq, 0, owq, 0, factor, np.arange(256))
    R.close()


def test_gemm_accumulation_all_positive_k16384(gpu_lib):
    """All-positive operands at K = 16384: the accumulated sum grows at every
    step, the hardest case for a reduced-precision accumulator."""
    rng = np.random.default_rng(11)
    M, N, K = 128, 256, 16384
    A = rng.integers(0x30, 0x48, (M, K)).astype(np.uint8)  # E4M3 in [0.5, 4)
    B = rng.integers(0x30, 0x48, (N, K)).astype(np.uint8)
    _full_check(gpu_lib, A, 0, B, 0, sa=1.0, sb=1.0)


def _te_operands(fp8, T, fin, fout, layer):
    """X, W, dY of one layer cast on the GPU (current scaling), with transposes."""
    x = synthetic.normal((T, fin), 1.0, synthetic.seed_for(3, layer, "x"), device="cuda")
    w = synthetic.normal((fout, fin), 0.02, synthetic.seed_for(3, layer, "w"), device="cuda")
    dy = synthetic.grad_like((T, fout), synthetic.seed_for(4, layer, "dy"), device="cuda")
    R = fp8.Recipe(4)
    xq, xt = R.quantize(0, x, fp8.E4M3, fp8.CURRENT, transpose=True)
    wq, wt = R.quantize(1, w, fp8.E4M3, fp8.CURRENT, transpose=True)
    dq, dt = R.quantize(2, dy, fp8.E5M2, fp8.CURRENT, transpose=True)
    return R, (xq, xt), (wq, wt), (dq, dt)


@pytest.mark.parametrize("layer", [0, 1, 2, 3])
def test_te_layer_gemms_sampled(gpu_lib, layer):
    fp8 = gpu_lib
    T = 8192
    _, fin, fout = synthetic.TE_LAYERS[layer]
    R, (xq, xt), (wq, wt), (dq, dt) = _te_operands(fp8, T, fin, fout, layer)
    rng = np.random.default_rng(100 + layer)
    sinv = [np.float32(R.get_state(t)[0]["cast_scale_inv"]) for t in range(3)]
    cases = [  # (name, A, afmt, a_id, B, bfmt, b_id)
        ("fwd", xq, 0, 0, wq, 0, 1),      # Y  [T, out]  = X  . W^T
        ("dgrad", dq, 1, 2, wt, 0, 1),    # dX [T, in]   = dY . W
        ("wgrad", dt, 1, 2, xt, 0, 0),    # dW [out, in] = dY^T . X
    ]
    for name, A, afmt, aid, B, bfmt, bid in cases:
        M, N = A.shape[0], B.shape[0]
        D32 = R.gemm(aid, A, afmt, bid, B, bfmt, out_dtype=fp8.OUT_F32)
        Db = R.gemm(aid, A, afmt, bid, B, bfmt)
        torch.cuda.synchronize()
        R.check_device_error()
        rows = np.sort(rng.choice(M, 256, replace=False))
        cols = np.sort(rng.choice(N, 256, replace=False))
        factor = sinv[aid] * sinv[bid]
        worst = check_gemm_sample(D32, Db, to_host_u8(A), afmt, to_host_u8(B), bfmt, factor, rows, cols)
        assert worst <= 1, name
        del D32, Db
    R.close()


def test_gemm_rejects_bad_k(gpu_lib):
    fp8 = gpu_lib
    R = fp8.Recipe(2)
    A = torch.zeros((16, 24), dtype=torch.uint8, device="cuda")
    with pytest.raises(fp8.Fp8Error) as e:
        R.gemm(0, A, 0, 1, A, 0)
    assert e.value.status == 1
    R.close()
