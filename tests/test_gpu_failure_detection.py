"""Failure detection without a GPU fault: a bounded device wait is made to run
out on purpose (fp8_debug_inject_stall over-states one shared-memory stage's
byte count, so the stage never completes -- the copy itself lands normally),
the kernel records the error and returns, the next synchronising call reports
FP8_ERR_TIMEOUT, and the same context then runs normal calls correctly."""
import numpy as np
import pytest
import torch

import oracle
from fp8_mixed_precision_history_gb300 import synthetic

pytestmark = pytest.mark.gpu

TIMEOUT = 4


def test_cast_wait_runs_out_and_is_reported(gpu_lib):
    fp8 = gpu_lib
    R = fp8.Recipe(1)
    x = synthetic.normal((1024, 1024), 1.0, 3)
    xd = x.cuda()
    fp8.fp8_debug_inject_stall(R.handle, fp8.STALL_CAST)
    R.quantize(0, xd, fp8.E4M3, fp8.CURRENT, transpose=True)  # the launch itself succeeds
    with pytest.raises(fp8.Fp8Error) as e:
        R.check_device_error()
    assert e.value.status == TIMEOUT and "cast" in str(e.value)
    R.check_device_error()  # reported once, then cleared
    # the context is intact: the same cast now matches the oracle bit for bit
    q, qt = R.quantize(0, xd, fp8.E4M3, fp8.CURRENT, transpose=True)
    torch.cuda.synchronize()
    R.check_device_error()
    xb = synthetic.bits(x)
    want, _, _ = oracle.cast(xb, oracle.scale_from_amax(oracle.amax(xb), oracle.E4M3), oracle.E4M3)
    assert np.array_equal(q.cpu().numpy(), want) and np.array_equal(qt.cpu().numpy(), want.T)
    R.close()


def test_gemm_wait_runs_out_and_is_reported(gpu_lib):
    """M = 512: the two-CTA kernel here (both CTAs of each pair leave through
    their bounded waits), the one-CTA kernel in test_gpu_gemm_one (which runs
    this file again with that kernel selected)."""
    fp8 = gpu_lib
    R = fp8.Recipe(2)
    rng = np.random.default_rng(1)
    A = oracle.encode(rng.standard_normal((512, 1024)) * 30, oracle.E4M3)
    B = oracle.encode(rng.standard_normal((384, 1024)) * 30, oracle.E4M3)
    R.set_state(0, [1.0] * 16, 1.0 / 64, 0)
    R.set_state(1, [1.0] * 16, 1.0 / 64, 0)
    Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    fp8.fp8_debug_inject_stall(R.handle, fp8.STALL_GEMM)
    R.gemm(0, Ad, 0, 1, Bd, 0, out_dtype=fp8.OUT_F32)  # the launch itself succeeds
    with pytest.raises(fp8.Fp8Error) as e:
        R.check_device_error()
    assert e.value.status == TIMEOUT and "gemm" in str(e.value)
    # the next GEMM on the same context is correct
    D = R.gemm(0, Ad, 0, 1, Bd, 0, out_dtype=fp8.OUT_F32)
    torch.cuda.synchronize()
    R.check_device_error()
    f = np.float32(64.0) * np.float32(64.0)  # 1/scale of each operand (scale 1/64), multiplied in fp32
    acc, absacc, _ = oracle.gemm(A, 0, B, 0, f, want_bf16=False)
    err = np.abs(D.cpu().numpy().astype(np.float64) - acc * float(f))
    assert np.all(err <= 1e-6 * absacc * float(f))
    R.close()


def test_inject_rejects_unknown_target(gpu_lib):
    fp8 = gpu_lib
    R = fp8.Recipe(1)
    with pytest.raises(fp8.Fp8Error):
        fp8.fp8_debug_inject_stall(R.handle, 7)
    R.close()
