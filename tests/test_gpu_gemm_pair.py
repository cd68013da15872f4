"""The two-CTA GEMM kernel (tcgen05.mma.cta_group::2, selected with
FP8LIN_GEMM_KERNEL=pair) against the oracle: the GEMM parity tests run again in
a fresh process with that kernel selected."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_pair_kernel_passes_gemm_parity(gpu_lib):
    env = dict(os.environ, FP8LIN_GEMM_KERNEL="pair")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
           os.path.join(HERE, "test_gpu_gemm.py"), "-k", "full_tensor or single_linear or strided or te_layer"]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


def test_pair_setting_runs_mn_major_calls_on_the_one_cta_kernel(gpu_lib):
    """The pair kernel reads K-major operands only; with it selected, calls with
    an MN-major operand run the one-CTA kernel and still meet the oracle."""
    env = dict(os.environ, FP8LIN_GEMM_KERNEL="pair")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
           os.path.join(HERE, "test_gpu_gemm_layout.py"), "-k", "strided or all_positive or te_layer"]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
