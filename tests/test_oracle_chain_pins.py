"""Pins of the oracle pieces the chained transformer-layer step adds (CPU).

* The MLP activation: the transformer layer of "4.2 Hopper I -- Transformer
  Engine / FP8" S4.2.6 (te.TransformerLayer, hidden 4096, FFN 16384) puts an
  activation between FC1 and FC2; the page does not name it, and the reading
  taken is GELU in its tanh form.  oracle.gelu / oracle.dgelu are pinned to
  PyTorch's own tanh-form GELU and its autograd derivative (float64 library
  routines), to the odd identity gelu(x) - gelu(-x) = x of that form, to the
  exact GELU x * Phi(x) it approximates, and to a finite difference.
* The next stage's cast composed into a GEMM epilogue (S4.2.4: the FP32 result
  is multiplied by 1/scale "or composed with the next stage's scale"):
  oracle.cast_f32 equals the pinned bf16 cast on bf16-valued inputs, and its
  counts and amax hold on inputs built to have known values.
* DelayedRecipe.record_cast: such a cast joins the tensor's history like any
  other cast of the step.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.recipe import DelayedRecipe


def _grid():
    return np.concatenate([np.linspace(-12.0, 12.0, 24001), [0.0, -0.0, 1e-30, -1e-30, 40.0, -40.0, 1e3, -1e3]])


def test_gelu_matches_torch_tanh_gelu():
    x = _grid()
    want = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    got = oracle.gelu(x)
    assert np.all(np.abs(got - want) <= 1e-14 * np.maximum(1.0, np.abs(x)))


def test_dgelu_matches_torch_autograd():
    x = _grid()
    xt = torch.from_numpy(x).requires_grad_(True)
    torch.nn.functional.gelu(xt, approximate="tanh").sum().backward()
    assert np.all(np.abs(oracle.dgelu(x) - xt.grad.numpy()) <= 1e-13)


def test_gelu_odd_identity_and_limits():
    """tanh is odd, so x/2 (1 + t(x)) - (-x)/2 (1 - t(x)) = x exactly."""
    x = np.linspace(-8.0, 8.0, 4001)
    assert np.all(np.abs(oracle.gelu(x) - oracle.gelu(-x) - x) <= 4e-16 * np.maximum(1.0, np.abs(x)))
    big = np.array([30.0, 1e4])
    assert np.array_equal(oracle.gelu(big), big) and np.all(oracle.gelu(-big) == 0.0)
    assert oracle.gelu(np.array([0.0]))[0] == 0.0
    assert np.all(oracle.dgelu(big) == 1.0) and np.all(oracle.dgelu(-big) == 0.0)
    assert oracle.dgelu(np.array([0.0]))[0] == 0.5


def test_gelu_tanh_form_approximates_x_phi():
    """The tanh form stays within 5e-4 of the exact GELU x * Phi(x) (its
    largest gap is about 4.7e-4, near |x| = 2); a wrong constant in sqrt(2/pi)
    or in the cubic term breaks this or the torch pin above."""
    from scipy.special import ndtr

    x = np.linspace(-10.0, 10.0, 40001)
    gap = np.abs(oracle.gelu(x) - x * ndtr(x))
    assert gap.max() < 5e-4
    assert gap.max() > 1e-4  # it is an approximation, not x * Phi(x) itself


def test_dgelu_is_the_derivative_of_gelu():
    x = np.linspace(-6.0, 6.0, 1201)
    h = 1e-5
    fd = (oracle.gelu(x + h) - oracle.gelu(x - h)) / (2 * h)
    assert np.all(np.abs(fd - oracle.dgelu(x)) <= 1e-8)


def test_cast_f32_equals_the_bf16_cast_on_bf16_values():
    rng = np.random.default_rng(3)
    xb = (rng.standard_normal(100_003).astype(np.float32) * 40).view(np.uint32)
    bits = (xb >> 16).astype(np.uint16)
    bits[::997] = 0x0000  # zeros
    for fmt, s in ((oracle.E4M3, 3.7), (oracle.E5M2, 1e-3), (oracle.E4M3, 11.0)):
        q1, ns1, nu1 = oracle.cast(bits, s, fmt)
        q2, ns2, nu2, am = oracle.cast_f32(oracle.bf16_to_f32(bits), s, fmt)
        assert np.array_equal(q1, q2) and (ns1, nu1) == (ns2, nu2)
        assert am == oracle.amax(bits)


def test_cast_f32_known_counts():
    """Four values saturate (|v*s| > 448, the last one is Inf), three
    underflow (nonzero, |v*s| <= 2^-10), zero is neither; amax is Inf."""
    v = np.array([500.0, -449.0, 448.0, 1e30, np.inf, 2.0 ** -11, -(2.0 ** -10), 2.0 ** -12, 0.0, 1.0,
                  2.0 ** -9], np.float32)
    q, ns, nu, am = oracle.cast_f32(v, 1.0, oracle.E4M3)
    assert ns == 4 and nu == 3 and np.isinf(am)
    assert list(q[:5]) == [0x7E, 0xFE, 0x7E, 0x7E, 0x7E]
    assert list(q[5:9]) == [0x00, 0x80, 0x00, 0x00] and q[10] == 0x01
    q, ns, nu, am = oracle.cast_f32(np.array([np.nan, 1.0], np.float32), 2.0, oracle.E5M2)
    assert np.isnan(am) and ns == 0 and nu == 0


def test_record_cast_joins_the_history():
    R = DelayedRecipe(1)
    R.set_state(0, [2.0] * 16, 224.0, oracle.E4M3)
    R.record_cast(0, np.float32(3.0), 5, 7, oracle.E4M3)
    R.record_cast(0, np.float32(1.5), 1, 0, oracle.E4M3)
    st = R.t[0]
    assert st.cast_scale == np.float32(224.0) and st.cast_scale_inv == oracle.reciprocal(224.0)
    assert st.amax_pending == np.float32(3.0) and (st.n_saturated, st.n_underflow) == (6, 7)
    R.update()
    assert st.history[-1] == np.float32(3.0) and st.scale == np.float32(448.0) / np.float32(3.0)
    assert (st.n_saturated_last, st.n_underflow_last) == (6, 7)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_cast_f32_ties_and_subnormals(fmt):
    """Every midpoint between neighbouring finite codes goes to the even code,
    through the fp32 product (scale 1: the product is the value itself)."""
    codes = np.arange(0, 0x7E if fmt == oracle.E4M3 else 0x7B, dtype=np.uint8)
    lo = oracle.decode(codes, fmt)
    hi = oracle.decode(codes + 1, fmt)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)  # exact in fp32
    q, _, _, _ = oracle.cast_f32(mid, 1.0, fmt)
    want = np.where(codes % 2 == 0, codes, codes + 1).astype(np.uint8)
    assert np.array_equal(q, want)
