"""The two-CTA MX GEMM kernel (selected with FP8LIN_MX_KERNEL=pair; by default
the one-CTA kernel runs every MX GEMM) against the oracle: the MX GEMM parity
tests of test_gpu_mx.py run again in a fresh process with that kernel
selected."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_pair_kernel_passes_mx_gemm_parity(gpu_lib):
    env = dict(os.environ, FP8LIN_MX_KERNEL="pair")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-k", "gemm or chain",
           os.path.join(HERE, "test_gpu_mx.py")]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " 0 passed" not in r.stdout
