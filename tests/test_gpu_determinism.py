"""Run twice, same bits: every kernel's result depends only on its inputs, not
on which CTA finished first.  The GEMMs add their TMEM partials in a fixed
order per tile (the split tail too), and every amax is an order-free max of
bit patterns; the MX quantiser and the all-reduce steps have no cross-CTA
arithmetic.  Each case compares two launches on fresh recipes: outputs,
recorded amax and counts."""
import numpy as np
import pytest
import torch

import oracle
from fp8_mixed_precision_history_gb300 import synthetic

pytestmark = pytest.mark.gpu

E4M3, E5M2 = oracle.E4M3, oracle.E5M2


def host(t):
    return t.contiguous().view(torch.uint8).cpu().numpy().copy()


@pytest.mark.parametrize("shape", [(8192, 4096, 4096), (300, 1000, 2320), (100, 520, 8192)])
@pytest.mark.parametrize("fp8_out", [False, True])
def test_gemm_twice(gpu_lib, shape, fp8_out):
    """Casts of X and W, then the GEMM: bf16 output with the output's amax
    recorded, or E4M3 output (its scale from tensor 2) with amax and counts."""
    fp8 = gpu_lib
    M, N, K = shape
    x = synthetic.normal((M, K), 1.0, 11).cuda()
    w = synthetic.normal((N, K), 0.02, 12).cuda()
    runs = []
    for _ in range(2):
        R = fp8.Recipe(3)
        xq = R.quantize(0, x, E4M3, fp8.CURRENT)
        wq = R.quantize(1, w, E4M3, fp8.CURRENT)
        d = R.gemm(0, xq, E4M3, 1, wq, E4M3, out_dtype=fp8.OUT_E4M3 if fp8_out else fp8.OUT_BF16,
                   amax_out_id=2)
        torch.cuda.synchronize()
        R.check_device_error()
        st, hist = R.get_state(2)
        runs.append((host(d), st, hist))
        R.close()
    assert np.array_equal(runs[0][0], runs[1][0]), "outputs differ between two runs"
    assert runs[0][1] == runs[1][1] and runs[0][2] == runs[1][2], "recorded state differs"


def test_mx_quantize_and_gemm_twice(gpu_lib):
    fp8 = gpu_lib
    M, N, K = 1024, 768, 4096
    a = synthetic.block_varied((M, K), 21).cuda()
    b = synthetic.block_varied((N, K), 22).cuda()
    runs = []
    for _ in range(2):
        R = fp8.Recipe(1)
        qa, sa, qat, sat = R.mx_quantize(a, E4M3, transpose=True)
        qb, sb = R.mx_quantize(b, E4M3)
        d = R.mx_gemm(qa, E4M3, sa, qb, E4M3, sb, out_dtype=fp8.OUT_F32)
        torch.cuda.synchronize()
        R.check_device_error()
        runs.append([host(t) for t in (qa, sa, qat, sat, qb, sb, d)])
        R.close()
    for name, u, v in zip(("q", "scales", "q^T", "scales^T", "B codes", "B scales", "D"), *runs):
        assert np.array_equal(u, v), f"{name} differs between two runs"


def test_all_reduce_twice(gpu_lib):
    from fp8_mixed_precision_history_gb300 import grad_allreduce

    world, n = 8, (1 << 20) + 3
    grads = [synthetic.grad_like((n,), 300 + r).cuda() for r in range(world)]
    runs = []
    for _ in range(2):
        out, codes = grad_allreduce.all_reduce_local(grads, average=True, with_codes=True)
        torch.cuda.synchronize()
        runs.append((host(out), host(codes)))
    assert np.array_equal(runs[0][0], runs[1][0]) and np.array_equal(runs[0][1], runs[1][1])
