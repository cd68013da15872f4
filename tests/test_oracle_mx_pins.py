"""Pins for the oracle's MX-style block scaling ("FP8 and low-precision formats",
format overview: per-tensor or per-block scale factors; MXFP8 elements share one
scale per block).

The pages give no rule for the block scale, so the oracle reads it as the
per-tensor rule restricted to powers of two ("4.2 Hopper I -- Transformer
Engine / FP8", S4.2.4: scale = FP8_MAX / amax): the largest 2^k, k in
[-127, 127], with amax_block * 2^k <= FP8_MAX.  These tests pin that reading and
the block partition with values worked out by hand, with brute force over all
codes, with exact rational sums and with the per-tensor GEMM it reduces to."""
from fractions import Fraction

import numpy as np
import pytest

import oracle

E4M3, E5M2 = oracle.E4M3, oracle.E5M2


def _bf16_bits(values):
    v = np.asarray(values, dtype=np.float32)
    bits = v.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "test values must be bf16-exact"
    return (bits >> 16).astype(np.uint16)


# (amax, format, k) worked out by hand: E4M3 max 448 = 1.75 * 2^8, E5M2 max
# 57344 = 1.75 * 2^15.
HAND = [
    (448.0, E4M3, 0),                 # exactly FP8_MAX
    (450.0, E4M3, -1),                # just above: 225 <= 448 < 450
    (1.0, E4M3, 8),                   # 256 <= 448 < 512
    (1.75, E4M3, 8),                  # 1.75 * 256 = 448 exactly
    (1.7578125, E4M3, 7),             # next bf16 above 1.75: 450 > 448
    (0.0, E4M3, 127),                 # empty block: the largest exponent
    (2.0 ** -133, E4M3, 127),         # smallest bf16 subnormal
    (2.0 ** -119, E4M3, 127),         # 2^-119 * 2^127 = 256 <= 448
    (2.0 ** -118, E4M3, 126),         # 2^9 = 512 > 448 at k = 127
    (1.9921875 * 2.0 ** 127, E4M3, -120),  # largest bf16: 1.99 * 2^7 = 255 <= 448, 2^8 * 1.99 > 448
    (float("inf"), E4M3, -127),
    (float("nan"), E4M3, -127),
    (57344.0, E5M2, 0),
    (1.0, E5M2, 15),                  # 32768 <= 57344 < 65536
    (1.9921875 * 2.0 ** 127, E5M2, -113),  # 1.99 * 2^14 = 32640 <= 57344 < 65280
]


@pytest.mark.parametrize("amax,fmt,k", HAND)
def test_mx_scale_exponent_worked_by_hand(amax, fmt, k):
    assert oracle.mx_scale_exponent(amax, fmt) == k


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_mx_scale_is_the_largest_power_of_two_that_fits(fmt):
    """amax * 2^k <= MAX < amax * 2^(k+1): exact in Python floats."""
    rng = np.random.default_rng(3)
    fmax = 448.0 if fmt == E4M3 else 57344.0
    bits = rng.integers(0x0080, 0x7F80, 4000).astype(np.uint16)  # normal bf16
    for b in bits:
        a = float(oracle.bf16_to_f32(np.array([b]))[0])
        k = oracle.mx_scale_exponent(a, fmt)
        assert a * 2.0 ** k <= fmax
        if k < 127:
            assert a * 2.0 ** (k + 1) > fmax


@pytest.mark.parametrize("fmt,top_code", [(E4M3, 0x7C), (E5M2, 0x7A)])
def test_mx_quantize_blocks_along_rows(fmt, top_code):
    """Block (r, b) holds smaller values plus one planted 1.5 * 2^(r-b) (negative
    in odd blocks).  Its exponent must be emax - (r - b), its scale code
    127 - k, and the planted element 1.5 * 2^emax (384 = 0x7C in E4M3, 49152 =
    0x7A in E5M2).  80 columns: the third block of each row has 16 elements."""
    emax = 8 if fmt == E4M3 else 15
    rows, cols = 5, 80
    rng = np.random.default_rng(11)
    x = np.zeros((rows, cols), dtype=np.float32)
    where = {}
    for r in range(rows):
        for b in range(3):
            c0, c1 = 32 * b, min(32 * b + 32, cols)
            top = 1.5 * 2.0 ** (r - b)
            small = rng.uniform(-1.0, 1.0, c1 - c0) * top
            x[r, c0:c1] = (small.astype(np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)
            p = c0 + int(rng.integers(0, c1 - c0))
            x[r, p] = -top if b % 2 else top
            where[(r, b)] = p
    q, sc = oracle.mx_quantize(_bf16_bits(x), fmt)
    assert sc.shape == (rows, 3)
    for (r, b), p in where.items():
        k = emax - (r - b)
        assert sc[r, b] == 127 - k
        assert q[r, p] == (top_code | (0x80 if b % 2 else 0))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_mx_codes_are_nearest_by_enumeration(fmt):
    """Each code is a nearest FP8 value of x * 2^k (ties to an even code),
    found here by enumerating all finite codes, not by the oracle's search."""
    rng = np.random.default_rng(5)
    rows, cols = 6, 96
    mag = np.exp(rng.uniform(np.log(1e-6), np.log(1e3), (rows, cols)))
    x = (mag * np.where(rng.random((rows, cols)) < 0.5, -1, 1)).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    xv = oracle.bf16_to_f32(bits).astype(np.float64)
    q, sc = oracle.mx_quantize(bits, fmt)
    finite = [c for c in range(256) if np.isfinite(oracle.decode(np.array([c]), fmt)[0])]
    vals = oracle.decode(np.array(finite, dtype=np.uint8), fmt)
    fmax = 448.0 if fmt == E4M3 else 57344.0
    for r in range(rows):
        for c in range(cols):
            k = 127 - int(sc[r, c // 32])
            v = xv[r, c] * 2.0 ** k
            assert abs(v) <= fmax  # the block scale never saturates
            d = np.abs(vals - v)
            best = d.min()
            got = oracle.decode(q[r:r + 1, c], fmt)[0]
            assert abs(got - v) == best
            if np.count_nonzero(d == best) > 1 and got != 0.0:
                assert q[r, c] % 2 == 0  # a tie went to the even mantissa
            if got == 0.0:
                assert (q[r, c] & 0x80) == (0x80 if v < 0 else 0)  # sign kept


def test_mx_gemm_with_uniform_scales_is_the_per_tensor_gemm():
    """With every block scale 2^sa and 2^sb the MX GEMM is the (pinned)
    per-tensor GEMM times 2^(sa+sb): a power-of-two factor is exact."""
    rng = np.random.default_rng(2)
    M, N, K = 7, 9, 100
    A = oracle.encode(rng.standard_normal((M, K)) * 30, E4M3)
    B = oracle.encode(rng.standard_normal((N, K)) * 3e3, E5M2)
    nb = (K + 31) // 32
    sa = np.full((M, nb), 127 - 5, np.uint8)
    sb = np.full((N, nb), 127 + 3, np.uint8)
    acc, ab, out = oracle.mx_gemm(A, E4M3, sa, B, E5M2, sb)
    ref, refab, _ = oracle.gemm(A, E4M3, B, E5M2, 1.0)
    assert np.array_equal(acc, ref * 2.0 ** -2)
    assert np.array_equal(ab, refab * 2.0 ** -2)
    assert np.array_equal(out, oracle.f64_to_bf16(ref * 2.0 ** -2))


def test_mx_gemm_exact_rational_sum():
    """Tiny MX GEMM with a different scale in every block (and a 6-element
    tail block) against an exact rational sum."""
    rng = np.random.default_rng(9)
    M, N, K = 3, 4, 70
    nb = 3
    A = rng.integers(0, 256, (M, K)).astype(np.uint8)
    B = rng.integers(0, 256, (N, K)).astype(np.uint8)
    A[(A & 0x7F) == 0x7F] = 0x11  # no NaN codes
    B[(B & 0x7F) == 0x7F] = 0x22
    sa = rng.integers(110, 145, (M, nb)).astype(np.uint8)
    sb = rng.integers(110, 145, (N, nb)).astype(np.uint8)
    acc, ab, _ = oracle.mx_gemm(A, E4M3, sa, B, E4M3, sb)
    da = oracle.decode(A, E4M3)
    db = oracle.decode(B, E4M3)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(da[m, k]) * Fraction(2) ** (int(sa[m, k // 32]) - 127)
                        * Fraction(db[n, k]) * Fraction(2) ** (int(sb[n, k // 32]) - 127) for k in range(K))
            mag = sum(abs(Fraction(da[m, k]) * Fraction(db[n, k])) * Fraction(2) ** (
                int(sa[m, k // 32]) + int(sb[n, k // 32]) - 254) for k in range(K))
            assert abs(Fraction(acc[m, n]) - exact) <= K * Fraction(2) ** -53 * mag
            assert abs(Fraction(ab[m, n]) - mag) <= K * Fraction(2) ** -53 * mag


def test_mx_gemm_block_scale_acts_on_its_block_only():
    """A single non-zero product in block j: the result is that product times
    the two scales of block j, whatever the other blocks' scales are."""
    M, N, K = 2, 2, 128
    A = np.zeros((M, K), np.uint8)
    B = np.zeros((N, K), np.uint8)
    A[1, 70] = 0x38  # 1.0 in E4M3
    B[0, 70] = 0x40  # 2.0
    sa = np.array([[127, 127, 127, 127], [100, 101, 120, 103]], np.uint8)
    sb = np.array([[131, 140, 135, 141], [127, 127, 127, 127]], np.uint8)
    acc, _, _ = oracle.mx_gemm(A, E4M3, sa, B, E4M3, sb)
    assert acc[1, 0] == 2.0 * 2.0 ** (120 - 127) * 2.0 ** (135 - 127)
    assert acc[0, 0] == 0.0 and acc[1, 1] == 0.0 and acc[0, 1] == 0.0


def test_e8m0_values():
    assert oracle.e8m0_value(127) == 1.0
    assert oracle.e8m0_value(0) == 2.0 ** -127
    assert oracle.e8m0_value(254) == 2.0 ** 127
    assert np.isnan(oracle.e8m0_value(255))
