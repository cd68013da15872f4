"""GPU parity of the delayed-scaling recipe (history roll and scale update)
against the oracle recipe, step by step and bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from oracle.recipe import ALGO_MOST_RECENT, DelayedRecipe
from fp8_mixed_precision_history_gb300 import synthetic
from gpu_util import check_state, to_host_u8

pytestmark = pytest.mark.gpu


def _drift_tensor(step, n=8192, spike_step=20):
    """Activation-like tensor whose std drifts x1.05 per step, x50 at the spike."""
    std = 1.05 ** step * (50.0 if step == spike_step else 1.0)
    return synthetic.normal((n,), std, seed=9000 + step)


@pytest.mark.parametrize("algo", [0, 1])
@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_history_loop_matches_oracle(gpu_lib, algo, fmt):
    R = gpu_lib.Recipe(3, amax_history_len=16, algo=algo)
    OR = DelayedRecipe(3, history_len=16, algo=algo)
    x0 = _drift_tensor(0)
    a0 = float(oracle.amax(synthetic.bits(x0)))
    s0 = float(oracle.scale_from_amax(a0, fmt))
    R.set_state(0, [a0] * 16, s0, fmt)
    OR.set_state(0, [a0] * 16, s0, fmt)
    for step in range(40):
        x = _drift_tensor(step)
        q = R.quantize(0, x.cuda(), fmt)
        oq = OR.quantize(0, synthetic.bits(x), fmt)
        assert np.array_equal(to_host_u8(q), oq), f"codes differ at step {step}"
        check_state(R, OR, 0, f"step {step} after cast")
        R.update_scales()
        OR.update()
        check_state(R, OR, 0, f"step {step} after update")
        check_state(R, OR, 1, f"step {step} untouched tensor")


def test_spike_saturates_then_underflows(gpu_lib):
    """The pages' qualitative claim: a spike is seen one step late."""
    R = gpu_lib.Recipe(1)
    sat, und = [], []
    n = 1 << 16
    x0 = _drift_tensor(0, n=n)
    a0 = float(oracle.amax(synthetic.bits(x0)))
    R.set_state(0, [a0] * 16, 448.0 / a0, gpu_lib.E4M3)
    for step in range(32):
        R.quantize(0, _drift_tensor(step, n=n).cuda(), gpu_lib.E4M3)
        R.update_scales()
        st, _ = R.get_state(0)
        sat.append(st["n_saturated_last"])
        und.append(st["n_underflow_last"])
    assert sat[20] > 100 and max(sat[:20]) < sat[20]
    assert min(und[21:]) > max(und[:20])


def test_update_touches_only_recorded(gpu_lib):
    R = gpu_lib.Recipe(4)
    OR = DelayedRecipe(4)
    x = synthetic.normal((1000,), 2.0, seed=1)
    R.quantize(2, x.cuda(), gpu_lib.E5M2)
    OR.quantize(2, synthetic.bits(x), oracle.E5M2)
    R.update_scales()
    OR.update()
    for t in range(4):
        check_state(R, OR, t, f"tensor {t}")


def test_checkpoint_resume_is_bit_identical(gpu_lib):
    xs = [_drift_tensor(s, n=4096) for s in range(12)]

    def run(R, steps):
        for s in steps:
            R.quantize(0, xs[s].cuda(), gpu_lib.E4M3)
            R.update_scales()

    A = gpu_lib.Recipe(1)
    run(A, range(12))
    B = gpu_lib.Recipe(1)
    run(B, range(7))
    st, hist = B.get_state(0)
    C = gpu_lib.Recipe(1)
    C.set_state(0, hist, st["scale"], gpu_lib.E4M3)
    run(C, range(7, 12))
    sa, ha = A.get_state(0)
    sc, hc = C.get_state(0)
    assert ha == hc and sa["scale"] == sc["scale"] and sa["scale_inv"] == sc["scale_inv"]


def test_set_state_validation(gpu_lib):
    R = gpu_lib.Recipe(1)
    with pytest.raises(gpu_lib.Fp8Error):
        R.set_state(0, [-1.0] * 16, 1.0, gpu_lib.E4M3)
    with pytest.raises(gpu_lib.Fp8Error):
        R.set_state(0, [1.0] * 16, 0.0, gpu_lib.E4M3)
    with pytest.raises(gpu_lib.Fp8Error):
        R.set_state(0, [float("nan")] * 16, 1.0, gpu_lib.E4M3)
    R.close()
