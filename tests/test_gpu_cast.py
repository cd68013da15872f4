"""GPU parity of the amax + scale + cast kernels against the CPU oracle.

Bit-exact on FP8 codes (and their transpose), amax, scales and the
saturation / underflow counts; covers one-pass delayed scaling, two-pass
current scaling, the fused history update, edge sizes and the standalone cast
sweep's distributions at 2^20, 2^24 and 2^28 elements."""
import numpy as np
import pytest
import torch

import oracle
from fp8_mixed_precision_history_gb300 import synthetic
from gpu_util import check_state, prefill_for, to_host_u8

pytestmark = pytest.mark.gpu

FMTS = [oracle.E4M3, oracle.E5M2]


def _cast_once(fp8, x, fmt, current, transpose=False, update_now=False, prefill_seed=None, draw=None):
    """Cast x (bf16 CPU tensor) on the GPU and in the oracle; compare.  With
    prefill_seed (delayed scaling) the history holds the amax of an independent
    draw(shape, prefill_seed), the previous step's tensor (default: spiky)."""
    xb = synthetic.bits(x)
    R = fp8.Recipe(1)
    OR = oracle.DelayedRecipe(1)
    if prefill_seed is not None:  # delayed scaling: history from an independent draw
        prev = (draw or synthetic.spiky)(x.shape, prefill_seed)
        hist, s = prefill_for(synthetic.bits(prev), fmt)
        R.set_state(0, hist, s, fmt)
        OR.set_state(0, hist, s, fmt)
    xd = x.cuda()
    mode = fp8.CURRENT if current else fp8.DELAYED
    res = R.quantize(0, xd, fmt, mode, update_now=update_now, transpose=transpose)
    torch.cuda.synchronize()
    R.check_device_error()
    q = res[0] if transpose else res
    oq = OR.quantize(0, xb, fmt, current=current, update_now=update_now)
    got = to_host_u8(q)
    mism = np.flatnonzero(got.reshape(-1) != oq.reshape(-1))
    assert mism.size == 0, f"{mism.size} codes differ, first at {mism[:5]}"
    if transpose:
        assert np.array_equal(to_host_u8(res[1]), oq.reshape(x.shape[0], -1).T)
    check_state(R, OR, 0, f"n={x.numel()}")
    R.close()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("current", [False, True])
@pytest.mark.parametrize("n", [1, 5, 16, 17, 255, 4099, 100003, 1 << 20])
def test_flat_cast_parity(gpu_lib, fmt, current, n):
    x = synthetic.spiky((n,), seed=2000 + n)
    _cast_once(gpu_lib, x, fmt, current, prefill_seed=None if current else 2001 + n)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(1, 16), (3, 17), (128, 128), (130, 200), (256, 4096),
                                   (1000, 48), (517, 1031), (16, 3000)])
def test_cast_transpose_parity(gpu_lib, fmt, shape):
    x = synthetic.normal(shape, 1.0, seed=3000 + shape[0] * 7 + shape[1])
    _cast_once(gpu_lib, x, fmt, current=False, transpose=True, prefill_seed=3001 + shape[1],
               draw=lambda sh, sd: synthetic.normal(sh, 1.0, sd))
    _cast_once(gpu_lib, x, fmt, current=True, transpose=True)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("current", [False, True])
def test_fused_update_now(gpu_lib, fmt, current):
    x = synthetic.spiky((50000,), seed=4000)
    _cast_once(gpu_lib, x, fmt, current, update_now=True, prefill_seed=None if current else 4001)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("current", [False, True])
@pytest.mark.parametrize("variant", ["spiky", "tiny"])
@pytest.mark.parametrize("log2n", [20, 24])
def test_cast_sweep_sizes(gpu_lib, fmt, current, variant, log2n):
    n = 1 << log2n
    seed = 1000 * 2 + log2n
    draw = _SWEEP_DRAW[variant]
    _cast_once(gpu_lib, draw((n,), seed), fmt, current, prefill_seed=None if current else seed + 1, draw=draw)


# the sweep's two distributions (a delayed cast's history comes from the same one)
_SWEEP_DRAW = {"spiky": synthetic.spiky, "tiny": lambda shape, seed: synthetic.normal(shape, 1e-3, seed)}


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("current", [False, True])
@pytest.mark.parametrize("variant", ["spiky", "tiny"])
def test_cast_sweep_2pow28(gpu_lib, fmt, current, variant):
    """The sweep's largest size in every variant: delayed (history from an
    independent draw) and current scaling, N(0,1) with 0.1 % spikes and the
    all-tiny N(0, 1e-3)."""
    n = 1 << 28
    seed = 1000 * 2 + 28
    draw = _SWEEP_DRAW[variant]
    _cast_once(gpu_lib, draw((n,), seed), fmt, current, prefill_seed=None if current else seed + 1, draw=draw)


@pytest.mark.parametrize("fmt", FMTS)
def test_tiny_tensor_after_spiky_history(gpu_lib, fmt):
    """A delayed cast whose history is far above the tensor (the step after a
    spike): most values flush to zero and are counted as underflowed."""
    n = (1 << 20) + 77
    _cast_once(gpu_lib, synthetic.normal((n,), 1e-3, 2031), fmt, False, prefill_seed=2032)


def test_special_values(gpu_lib):
    vals = [0.0, -0.0, 1.0, -1.0, 3e38, -3e38, float("inf"), -float("inf"), 1e-40, -1e-40,
            448.0, 464.0, 57344.0, 61440.0, 2.0 ** -10, -(2.0 ** -10), 2.0 ** -17, 2.0 ** -9]
    x = torch.tensor(vals * 3, dtype=torch.float32).to(torch.bfloat16)
    for fmt in FMTS:
        R = gpu_lib.Recipe(1)
        OR = oracle.DelayedRecipe(1)
        q = R.quantize(0, x.cuda(), fmt)
        oq = OR.quantize(0, synthetic.bits(x), fmt)
        assert np.array_equal(to_host_u8(q), oq)
        check_state(R, OR, 0, "special")
        R.close()


def test_determinism(gpu_lib):
    x = synthetic.spiky((3_000_001,), seed=5)
    xd = x.cuda()
    outs = []
    for _ in range(2):
        R = gpu_lib.Recipe(1)
        q = R.quantize(0, xd, gpu_lib.E4M3, gpu_lib.CURRENT)
        st, _ = R.get_state(0)
        outs.append((to_host_u8(q), st))
        R.close()
    assert np.array_equal(outs[0][0], outs[1][0]) and outs[0][1] == outs[1][1]


def test_e4m3_recipe_rejects_e5m2(gpu_lib):
    R = gpu_lib.Recipe(1, format=gpu_lib.RECIPE_E4M3)
    x = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(gpu_lib.Fp8Error):
        R.quantize(0, x, gpu_lib.E5M2)
    R.close()


def test_unaligned_pointer_rejected(gpu_lib):
    R = gpu_lib.Recipe(1)
    x = torch.zeros(100, dtype=torch.bfloat16, device="cuda")
    q = torch.empty(100, dtype=torch.uint8, device="cuda")
    with pytest.raises(gpu_lib.Fp8Error) as e:
        gpu_lib.fp8_amax_quantize(R.handle, 0, x.data_ptr() + 2, 1, 16, gpu_lib.E4M3,
                                  gpu_lib.DELAYED, 0, q, None)
    assert e.value.status == 1
    R.close()
