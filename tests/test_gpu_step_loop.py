"""The 32-step delayed-scaling training loop ("4.2 Hopper I -- Transformer
Engine / FP8", S4.2.4 delayed scaling and S4.2.6 recipe: history of 16, "max").

Per step, for each of the four linear layers: cast X and W (E4M3), forward
GEMM with the output amax fused into the epilogue, cast dY (E5M2), dgrad and
wgrad on the same codes read MN-major (no transposed copies); then one scale
update.  Activations drift x1.05 per
step and spike x50 at step 20; weights are fixed; gradients are fresh each step.

* At reduced size every tensor's state (amax, scales, counts, history) is
  compared with the oracle recipe after every step, bit for bit.
* At full size (16384 tokens, hidden 4096, FFN 16384) the oracle follows
  layer 0's activation tensor through every step (bit for bit), and every
  layer's reported state is checked for the relations that hold at any size.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.recipe import DelayedRecipe
from fp8_mixed_precision_history_gb300 import synthetic
from gpu_util import check_state, f32_bits

pytestmark = pytest.mark.gpu

STEPS = 32
SPIKE = 20


def _x(step, li, T, fin, device):
    std = 1.05 ** step * (50.0 if step == SPIKE else 1.0)
    return synthetic.normal((T, fin), std, synthetic.seed_for(5, li, "x", step), device=device)


def _w(li, fin, fout, device):
    return synthetic.normal((fout, fin), 0.02, synthetic.seed_for(5, li, "w"), device=device)


def _dy(step, li, T, fout, device):
    return synthetic.grad_like((T, fout), synthetic.seed_for(5, li, "dy", step), device=device)


def _run_step(fp8, R, step, layers, T, device, W, bufs, gen_device=None):
    """One training step through the C ABI; returns the forward outputs.
    Inputs are drawn on gen_device (default: device) and moved to device."""
    gen = gen_device or device
    ys = []
    for li, (_, fin, fout) in enumerate(layers):
        x = _x(step, li, T, fin, gen).to(device)
        xq = R.quantize(4 * li, x, fp8.E4M3)
        wq = R.quantize(4 * li + 1, W[li], fp8.E4M3)
        y = R.gemm(4 * li, xq, fp8.E4M3, 4 * li + 1, wq, fp8.E4M3, amax_out_id=4 * li + 3)
        dy = _dy(step, li, T, fout, gen).to(device)
        dq = R.quantize(4 * li + 2, dy, fp8.E5M2)
        R.gemm(4 * li + 2, dq, fp8.E5M2, 4 * li + 1, wq, fp8.E4M3, b_major=fp8.MN_MAJOR)   # dgrad
        R.gemm(4 * li + 2, dq, fp8.E5M2, 4 * li, xq, fp8.E4M3, a_major=fp8.MN_MAJOR,
               b_major=fp8.MN_MAJOR)                                                       # wgrad
        bufs[li] = (x, dy)
        ys.append(y)
    return ys


def test_loop_reduced_size_matches_oracle(gpu_lib):
    fp8 = gpu_lib
    T = 256
    layers = (("qkv", 128, 384), ("proj", 128, 128), ("fc1", 128, 512), ("fc2", 512, 128))
    dev = torch.device("cuda")
    R = fp8.Recipe(4 * len(layers))
    OR = DelayedRecipe(4 * len(layers))
    W = [_w(li, fin, fout, "cpu") for li, (_, fin, fout) in enumerate(layers)]
    Wd = [w.to(dev) for w in W]
    # warm start: histories pre-filled with each tensor's step-0 amax
    for li, (_, fin, fout) in enumerate(layers):
        for tid, t, fmt in ((4 * li, _x(0, li, T, fin, "cpu"), 0), (4 * li + 1, W[li], 0),
                            (4 * li + 2, _dy(0, li, T, fout, "cpu"), 1)):
            a = float(oracle.amax(synthetic.bits(t)))
            s = float(oracle.scale_from_amax(a, fmt))
            R.set_state(tid, [a] * 16, s, fmt)
            OR.set_state(tid, [a] * 16, s, fmt)
    bufs = [None] * len(layers)
    for step in range(STEPS):
        _run_step(fp8, R, step, layers, T, dev, Wd, bufs, gen_device="cpu")
        for li, (_, fin, fout) in enumerate(layers):
            xq = OR.quantize(4 * li, synthetic.bits(_x(step, li, T, fin, "cpu")), 0)
            wq = OR.quantize(4 * li + 1, synthetic.bits(W[li]), 0)
            OR.quantize(4 * li + 2, synthetic.bits(_dy(step, li, T, fout, "cpu")), 1)
            # forward output amax from the oracle's own GEMM
            f = np.float32(OR.t[4 * li].cast_scale_inv) * np.float32(OR.t[4 * li + 1].cast_scale_inv)
            _, _, yb = oracle.gemm(xq, 0, wq, 0, f, want_abs=False)
            OR.record_amax(4 * li + 3, np.max(np.abs(oracle.bf16_to_f32(yb))))
        for tid in range(4 * len(layers)):
            if tid % 4 == 3:
                _check_output_amax(R, OR, tid, f"step {step}")
            else:
                check_state(R, OR, tid, f"step {step} before update")
        R.update_scales()
        OR.update()
        for tid in range(4 * len(layers)):
            if tid % 4 != 3:
                check_state(R, OR, tid, f"step {step} after update")
    R.close()


def _check_output_amax(R, OR, tid, what):
    """A GEMM-epilogue amax: the GPU's output may sit 1 bf16 ulp from the
    oracle's rounding, so its amax is compared within 1 ulp."""
    st, _ = R.get_state(tid)
    g = f32_bits(st["amax_pending"]) >> 16
    o = f32_bits(OR.t[tid].amax_pending) >> 16
    assert abs(g - o) <= 1 and (f32_bits(st["amax_pending"]) & 0xFFFF) == 0, what
    assert bool(st["recorded"]) and bool(OR.t[tid].recorded), what


def test_loop_full_size_properties(gpu_lib):
    fp8 = gpu_lib
    T = 16384
    layers = synthetic.TE_LAYERS
    dev = torch.device("cuda")
    R = fp8.Recipe(4 * len(layers))
    OR = DelayedRecipe(1)  # the oracle follows layer 0's activations through every step
    W = [_w(li, fin, fout, dev) for li, (_, fin, fout) in enumerate(layers)]
    # warm start from a current-scaling pass over step 0's tensors
    for li, (_, fin, fout) in enumerate(layers):
        x0 = _x(0, li, T, fin, dev)
        R.quantize(4 * li, x0, fp8.E4M3, fp8.CURRENT)
        if li == 0:
            OR.quantize(0, synthetic.bits(x0), oracle.E4M3, current=True)
        R.quantize(4 * li + 1, W[li], fp8.E4M3, fp8.CURRENT)
        R.quantize(4 * li + 2, _dy(0, li, T, fout, dev), fp8.E5M2, fp8.CURRENT)
    R.update_scales()
    OR.update()
    bufs = [None] * len(layers)
    sat = np.zeros((STEPS, len(layers)), np.int64)
    und = np.zeros((STEPS, len(layers)), np.int64)
    for step in range(STEPS):
        _run_step(fp8, R, step, layers, T, dev, W, bufs)
        OR.quantize(0, synthetic.bits(bufs[0][0]), oracle.E4M3)
        check_state(R, OR, 0, f"step {step} layer-0 activations")
        R.update_scales()
        OR.update()
        check_state(R, OR, 0, f"step {step} layer-0 activations after update")
        for li in range(len(layers)):
            st, hist = R.get_state(4 * li)
            sat[step, li] = st["n_saturated_last"]
            und[step, li] = st["n_underflow_last"]
            # scale for the next step = 448 / max(history), fp32 division
            m = np.float32(max(hist))
            assert f32_bits(st["scale"]) == f32_bits(np.float32(448.0) / m), (step, li)
            assert hist[-1] == st["amax_last"]
    R.check_device_error()
    R.close()
    # the spike is seen one step late: its own step saturates (the steady x1.05
    # drift saturates a handful of tail values per step, the spike most values)
    assert (sat[SPIKE] > 1000 * np.maximum(1, sat[:SPIKE].max(axis=0))).all()
    # for the 16 steps the spike stays in the history, small values flush to zero
    base = und[SPIKE - 4:SPIKE].mean(axis=0)
    assert (und[SPIKE + 1:SPIKE + 12].min(axis=0) > 2 * base).all()
