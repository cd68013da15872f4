"""The one-CTA GEMM kernel (selected with FP8LIN_GEMM_KERNEL=one; by default it
runs only when M <= 128, and the two-CTA kernel takes larger M) against the
oracle: the GEMM parity tests, including the FP8-output epilogue, MN-major
operands, the fused activation and the injected time-out, run again in a fresh process with that
kernel selected."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_one_cta_kernel_passes_gemm_parity(gpu_lib):
    env = dict(os.environ, FP8LIN_GEMM_KERNEL="one")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
           os.path.join(HERE, "test_gpu_gemm.py"), os.path.join(HERE, "test_gpu_gemm_fp8_out.py"),
           os.path.join(HERE, "test_gpu_gemm_layout.py"), os.path.join(HERE, "test_gpu_failure_detection.py"),
           os.path.join(HERE, "test_gpu_gemm_act.py")]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
