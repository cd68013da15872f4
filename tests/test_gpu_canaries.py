"""Guard bytes after every output: each kernel writes its output and nothing
past it.  Every output is a view at the start of a larger buffer filled with
0xAB; the sizes are ragged, so the last vector, block or tile of each kernel
is partial.  After the call the bytes past the output must still be 0xAB.
(compute-sanitizer is not available here; these checks stand in for its
out-of-bounds write detection on the outputs.)"""
import numpy as np
import pytest
import torch

import oracle
from fp8_mixed_precision_history_gb300 import synthetic

pytestmark = pytest.mark.gpu

E4M3, E5M2 = oracle.E4M3, oracle.E5M2
GUARD = 256


def guarded(nbytes):
    """(buffer, uint8 view of its first nbytes); the buffer is 16-byte aligned."""
    buf = torch.full((nbytes + GUARD,), 0xAB, dtype=torch.uint8, device="cuda")
    return buf, buf[:nbytes]


def assert_guard(buf, nbytes, what):
    torch.cuda.synchronize()
    tail = buf[nbytes:].cpu().numpy()
    bad = int((tail != 0xAB).sum())
    assert bad == 0, f"{what}: {bad} of the {GUARD} guard bytes were written"


def codes(shape, seed):
    """Finite E4M3/E5M2 codes (exponent field below all ones)."""
    rng = np.random.default_rng(seed)
    c = rng.integers(0, 256, size=shape, dtype=np.uint8) & np.uint8(0xBB)  # clears a high exponent bit
    return torch.from_numpy(c).cuda()


@pytest.mark.parametrize("n", [1, 7, 9, 4099, (1 << 20) + 5])
@pytest.mark.parametrize("mode", ["delayed", "current"])
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_cast(gpu_lib, n, mode, fmt):
    fp8 = gpu_lib
    x = synthetic.normal((n,), 1.0, 40 + n).cuda()
    buf, out = guarded(n)
    R = fp8.Recipe(1)
    R.quantize(0, x, fmt, mode=fp8.DELAYED if mode == "delayed" else fp8.CURRENT, out=out)
    R.check_device_error()
    R.close()
    assert_guard(buf, n, f"cast of {n}")


@pytest.mark.parametrize("shape", [(130, 144), (129, 131), (8, 16), (257, 1040)])
def test_cast_transpose(gpu_lib, shape):
    """cols % 8 == 0 takes the TMA kernel, other widths the register kernel."""
    fp8 = gpu_lib
    rows, cols = shape
    x = synthetic.normal(shape, 1.0, rows + cols).cuda()
    qbuf, q = guarded(rows * cols)
    tbuf, qt = guarded(rows * cols)
    R = fp8.Recipe(1)
    R.quantize(0, x, E4M3, transpose=True, out=q.view(rows, cols), out_t=qt.view(cols, rows))
    R.check_device_error()
    R.close()
    assert_guard(qbuf, rows * cols, f"codes of {shape}")
    assert_guard(tbuf, rows * cols, f"transposed codes of {shape}")


def test_cast_without_allocation(gpu_lib):
    fp8 = gpu_lib
    n = 70001
    x = synthetic.normal((n,), 1.0, 5).cuda()
    buf, out = guarded(n)
    sbuf, sc = guarded(8)
    cbuf, cnt = guarded(16)
    fp8.fp8_quantize_current_noalloc(x, n, E5M2, out, sc.view(torch.float32), cnt.view(torch.int64))
    assert_guard(buf, n, "codes")
    assert_guard(sbuf, 8, "scale pair")
    assert_guard(cbuf, 16, "counts")


@pytest.mark.parametrize("shape", [(304, 1008), (144, 160), (300, 1008)])
def test_mx_quantize(gpu_lib, shape):
    """With the transposed copy where rows % 16 == 0 allows it."""
    fp8 = gpu_lib
    rows, cols = shape
    x = synthetic.block_varied(shape, rows * cols % 997).cuda()
    transpose = rows % 16 == 0
    qbuf, q = guarded(rows * cols)
    sbytes = fp8.fp8_mx_scale_bytes(rows, cols)
    sbuf, qs = guarded(sbytes)
    R = fp8.Recipe(1)
    if transpose:
        tbuf, qt = guarded(rows * cols)
        tsbytes = fp8.fp8_mx_scale_bytes(cols, rows)
        tsbuf, qts = guarded(tsbytes)
        fp8.fp8_mx_quantize(R.handle, x, rows, cols, E4M3, q, qs, qt, qts)
    else:
        fp8.fp8_mx_quantize(R.handle, x, rows, cols, E4M3, q, qs)
    R.check_device_error()
    R.close()
    assert_guard(qbuf, rows * cols, "codes")
    assert_guard(sbuf, sbytes, "block scales")
    if transpose:
        assert_guard(tbuf, rows * cols, "transposed codes")
        assert_guard(tsbuf, tsbytes, "transposed block scales")


@pytest.mark.parametrize("out", ["bf16", "f32", "e4m3"])
@pytest.mark.parametrize("shape", [(300, 264, 208), (100, 264, 208), (100, 136, 6160), (1000, 520, 2048)])
def test_gemm(gpu_lib, out, shape):
    """M > 128 runs the two-CTA kernel, M <= 128 the one-CTA kernel, or on a
    long K the two-CTA kernel with every tile split.  Rows whose width is not
    a multiple of 16 bytes take the direct stores instead of TMA."""
    fp8 = gpu_lib
    M, N, K = shape
    A, B = codes((M, K), M + K), codes((N, K), N + K + 1)
    kind, esize, dt = {"bf16": (fp8.OUT_BF16, 2, torch.bfloat16), "f32": (fp8.OUT_F32, 4, torch.float32),
                       "e4m3": (fp8.OUT_E4M3, 1, torch.uint8)}[out]
    buf, d = guarded(M * N * esize)
    R = fp8.Recipe(3)
    R.gemm(0, A, E4M3, 1, B, E4M3, out_dtype=kind, out=d.view(dt).view(M, N),
           amax_out_id=2 if out == "e4m3" else -1)
    R.check_device_error()
    R.close()
    assert_guard(buf, M * N * esize, f"{out} output of {shape}")


@pytest.mark.parametrize("shape", [(300, 1000, 208), (1024, 272, 4096)])
def test_mx_gemm(gpu_lib, shape):
    fp8 = gpu_lib
    M, N, K = shape
    R = fp8.Recipe(1)
    qa, sa = R.mx_quantize(synthetic.block_varied((M, K), 1).cuda(), E4M3)
    qb, sb = R.mx_quantize(synthetic.block_varied((N, K), 2).cuda(), E4M3)
    buf, d = guarded(M * N * 2)
    R.mx_gemm(qa, E4M3, sa, qb, E4M3, sb, out=d.view(torch.bfloat16).view(M, N))
    R.check_device_error()
    R.close()
    assert_guard(buf, M * N * 2, f"MX GEMM output of {shape}")


@pytest.mark.parametrize("world", [3, 8, 200])
def test_grad_reduce_and_dequantize(gpu_lib, world):
    fp8 = gpu_lib
    chunk = 4096 + 16
    recv = codes((world, chunk), world)
    buf, out = guarded(chunk)
    fp8.fp8_grad_reduce(recv, world, chunk, out)
    assert_guard(buf, chunk, f"reduced codes, world {world}")
    n = chunk - 9
    scale = torch.tensor([2.0, 0.5], dtype=torch.float32, device="cuda")
    dbuf, d = guarded(2 * n)
    fp8.fp8_grad_dequantize(out, n, scale, world, True, d.view(torch.bfloat16))
    assert_guard(dbuf, 2 * n, f"dequantised output, world {world}")
