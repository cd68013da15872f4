"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Every test here runs on CPU.  The expected values come from the pages (golden
fixtures with citations), from the OCP FP8 definition the pages name, from
independent library routines (torch's float8 / bf16 dtypes, numpy float16),
from exact rational arithmetic, or from inputs built so that the answer is
known by construction.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
E4M3, E5M2 = 0, 1
FMT = {"e4m3": E4M3, "e5m2": E5M2}
TORCH_FP8 = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def _bf16_bits(vals):
    t = torch.tensor(np.asarray(vals, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- decode ----

def test_decode_ocp_points(oracle_mod):
    n = 0
    for fmt, code, val in _rows("ocp_fp8_points.txt"):
        got = oracle_mod.decode(np.array([int(code, 16)], np.uint8), FMT[fmt])[0]
        if val == "nan":
            assert math.isnan(got), (fmt, code)
        else:
            want = float(val)
            assert got == want, (fmt, code, got, want)
            assert math.copysign(1.0, got) == math.copysign(1.0, want), (fmt, code)
        n += 1
    assert n >= 30


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_decode_all_codes_match_torch_float8(oracle_mod, fmt):
    c = np.arange(256, dtype=np.uint8)
    got = oracle_mod.decode(c, fmt)
    ref = torch.from_numpy(c).view(TORCH_FP8[fmt]).to(torch.float64).numpy()
    assert np.array_equal(got, ref, equal_nan=True)
    fin = ~np.isnan(ref)
    assert np.array_equal(np.signbit(got[fin]), np.signbit(ref[fin]))  # -0 included


def test_e5m2_decode_is_top_byte_of_binary16(oracle_mod):
    # E5M2 shares binary16's exponent field: code c is the half-float c << 8.
    c = np.arange(256, dtype=np.uint8)
    half = (c.astype(np.uint16) << 8).view(np.float16).astype(np.float64)
    assert np.array_equal(oracle_mod.decode(c, E5M2), half, equal_nan=True)


def test_max_finite(oracle_mod):
    assert oracle_mod.fp8_max(E4M3) == 448.0
    assert oracle_mod.fp8_max(E5M2) == 57344.0
    v = oracle_mod.decode(np.arange(256, dtype=np.uint8), E4M3)
    assert np.nanmax(np.abs(v)) == 448.0 and not np.isinf(v).any()
    v = oracle_mod.decode(np.arange(256, dtype=np.uint8), E5M2)
    assert np.max(np.abs(v[np.isfinite(v)])) == 57344.0


# ---------------------------------------------------------------- encode ----

@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_roundtrip_every_code(oracle_mod, fmt):
    c = np.arange(256, dtype=np.uint8)
    v = oracle_mod.decode(c, fmt)
    ok = np.isfinite(v)
    back = oracle_mod.encode(v[ok].astype(np.float32), fmt)
    assert np.array_equal(back, c[ok])  # +0 -> 0x00 and -0 -> 0x80 stay distinct


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_matches_torch_in_range(oracle_mod, fmt):
    mx = oracle_mod.fp8_max(fmt)
    rng = np.random.default_rng(7)
    # log-uniform magnitudes over the whole range incl. subnormals and below
    e = rng.uniform(math.log2(mx) - 30, math.log2(mx), 200000)
    v = (np.exp2(e) * rng.choice([-1.0, 1.0], e.size)).astype(np.float32)
    v = v[np.abs(v) <= mx]
    # add exact midpoints between neighbouring codes (ties)
    pos = oracle_mod.decode(np.arange(128, dtype=np.uint8), fmt)
    pos = pos[np.isfinite(pos)]
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids])
    ref = torch.from_numpy(v).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
    assert np.array_equal(oracle_mod.encode(v, fmt), ref)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_ties_go_to_even_code(oracle_mod, fmt):
    pos = oracle_mod.decode(np.arange(128, dtype=np.uint8), fmt)
    top = 0x7E if fmt == E4M3 else 0x7B
    for c in range(top):
        mid = np.float32((pos[c] + pos[c + 1]) / 2)
        assert float(mid) == (pos[c] + pos[c + 1]) / 2  # exact in fp32
        want = c if c % 2 == 0 else c + 1
        assert oracle_mod.encode(np.array([mid]), fmt)[0] == want
        assert oracle_mod.encode(np.array([-mid]), fmt)[0] == 0x80 | want
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(np.inf))
        assert oracle_mod.encode(np.array([below]), fmt)[0] == c
        assert oracle_mod.encode(np.array([above]), fmt)[0] == c + 1


def test_encode_saturates_and_nan(oracle_mod):
    big = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, 3.4e38, np.inf], np.float32)
    assert list(oracle_mod.encode(big, E4M3)) == [0x7E] * big.size
    assert list(oracle_mod.encode(-big, E4M3)) == [0xFE] * big.size
    big5 = np.array([57344.0, 61439.0, 61440.0, 1e9, np.inf], np.float32)
    assert list(oracle_mod.encode(big5, E5M2)) == [0x7B] * big5.size
    assert list(oracle_mod.encode(-big5, E5M2)) == [0xFB] * big5.size
    nan = np.array([np.nan], np.float32)
    assert math.isnan(oracle_mod.decode(oracle_mod.encode(nan, E4M3), E4M3)[0])
    assert math.isnan(oracle_mod.decode(oracle_mod.encode(nan, E5M2), E5M2)[0])


@pytest.mark.parametrize("fmt,sub", [(E4M3, 2.0 ** -9), (E5M2, 2.0 ** -16)])
def test_encode_underflow_keeps_sign(oracle_mod, fmt, sub):
    v = np.array([sub / 2, np.nextafter(np.float32(sub / 2), np.float32(1)), sub * 0.25, 1e-30,
                  -sub / 2, -1e-30, -0.0, 0.0], np.float32)
    assert list(oracle_mod.encode(v, fmt)) == [0x00, 0x01, 0x00, 0x00, 0x80, 0x80, 0x80, 0x00]


# ------------------------------------------------------------------ bf16 ----

def test_bf16_rounding_matches_torch(oracle_mod):
    rng = np.random.default_rng(3)
    e = rng.uniform(-140, 127.9, 300000)
    v = (np.exp2(e) * rng.choice([-1.0, 1.0], e.size)).astype(np.float32)
    # bf16 midpoints: a bf16 value plus half its ulp (exact ties)
    b = _bf16_bits(v[:5000]).astype(np.uint32)
    base = (b << 16).view(np.float32)
    nxt = ((b + 1) << 16).view(np.float32)
    ties = ((base.astype(np.float64) + nxt.astype(np.float64)) / 2).astype(np.float32)
    v = np.concatenate([v, ties[np.isfinite(ties)]])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle_mod.f64_to_bf16(v.astype(np.float64)), ref)


def test_bf16_rounding_of_wide_values(oracle_mod):
    one = 1.0
    ulp = 2.0 ** -7
    cases = [
        (one, 0x3F80),
        (one + ulp / 2, 0x3F80),                    # tie -> even (1.0)
        (one + ulp / 2 + 2 ** -40, 0x3F81),         # just above the tie (not an fp32 value)
        (one + 1.5 * ulp, 0x3F82),                  # tie -> even (1 + 2 ulp)
        (-(one + ulp / 2 + 2 ** -40), 0xBF81),
        (3.3895313892515355e38, 0x7F7F),            # bf16 max
        (3.3961775292304744e38, 0x7F80),            # at the overflow tie -> Inf
        (1e300, 0x7F80),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (2.0 ** -133, 0x0001),                      # smallest bf16 subnormal
        (2.0 ** -134, 0x0000),                      # tie with 0 -> even (0)
        (2.0 ** -134 + 2.0 ** -160, 0x0001),
    ]
    for y, want in cases:
        assert oracle_mod.f64_to_bf16(np.array([y]))[0] == want, y


# ------------------------------------------------------------------ amax ----

def test_amax_matches_numpy(oracle_mod):
    rng = np.random.default_rng(11)
    x = _bf16_bits(rng.standard_normal(100003) * 3)
    want = np.max(np.abs((x.astype(np.uint32) << 16).view(np.float32)))
    assert oracle_mod.amax(x) == want
    assert oracle_mod.amax(_bf16_bits([0.0, -0.0])) == 0.0
    assert oracle_mod.amax(_bf16_bits([-5.0, 2.0])) == 5.0
    assert math.isnan(oracle_mod.amax(_bf16_bits([1.0, np.nan, 3.0])))
    assert oracle_mod.amax(_bf16_bits([1.0, -np.inf])) == np.inf


# ------------------------------------------------------------------ cast ----

@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_cast_equals_torch_cast_of_fp32_product(oracle_mod, fmt):
    rng = np.random.default_rng(5)
    x = _bf16_bits(rng.standard_normal(50000) * 0.7)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    s = np.float32(oracle_mod.fp8_max(fmt) / 4.1)
    q, ns, _ = oracle_mod.cast(x, s, fmt)
    p = torch.from_numpy(xf) * torch.tensor(s)  # fp32 products
    inr = p.abs() <= oracle_mod.fp8_max(fmt)
    ref = p.to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
    assert np.array_equal(q[inr.numpy()], ref[inr.numpy()])
    assert ns == int((~inr).sum())


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_cast_counts_by_construction(oracle_mod, fmt):
    mx = oracle_mod.fp8_max(fmt)
    sub = 2.0 ** -9 if fmt == E4M3 else 2.0 ** -16
    scale = np.float32(2.0)
    n_big, n_tiny, n_zero, n_mid = 37, 53, 11, 999
    vals = ([mx] * n_big                       # x*scale = 2*MAX: saturate
            + [sub / 8] * n_tiny               # x*scale = sub/4: flushed to 0
            + [0.0] * n_zero                   # zeros are not underflow
            + [1.0] * n_mid)                   # plain values
    vals = np.array(vals, np.float32) * np.where(np.arange(len(vals)) % 2, -1, 1)
    x = _bf16_bits(vals)
    q, ns, nu = oracle_mod.cast(x, scale, fmt)
    assert ns == n_big and nu == n_tiny
    top = 0x7E if fmt == E4M3 else 0x7B
    assert set(q[:n_big] & 0x7F) == {top}
    assert set(q[n_big:n_big + n_tiny + n_zero] & 0x7F) == {0}


# ----------------------------------------------------------------- scale ----

def test_worked_example_scales(oracle_mod):
    seen = 0
    for row in _rows("worked_example_scales.txt"):
        if row[0] == "range":
            lo, hi, want_lo, want_hi, tol = map(float, row[1:])
            s = oracle_mod.scale_from_amax(np.float32(hi), E4M3)
            assert abs(float(np.float32(lo) * s) - want_lo) <= tol
            assert abs(float(np.float32(hi) * s) - want_hi) <= tol
        else:
            a, want, tol = map(float, row)
            s = oracle_mod.scale_from_amax(np.float32(a), E4M3)
            assert abs(float(s) - want) <= tol, (a, s, want)
        seen += 1
    assert seen == 5


def _fp32_ulp(x):
    return float(np.spacing(np.float32(abs(x))))


def test_scale_is_correctly_rounded_division(oracle_mod):
    rng = np.random.default_rng(9)
    for fmt in (E4M3, E5M2):
        mx = Fraction(oracle_mod.fp8_max(fmt))
        for a in np.exp2(rng.uniform(-30, 30, 2000)).astype(np.float32):
            s = oracle_mod.scale_from_amax(a, fmt)
            exact = mx / Fraction(float(a))
            err = abs(Fraction(float(s)) - exact)
            assert err <= Fraction(_fp32_ulp(s)) / 2, (a, s)
            r = oracle_mod.reciprocal(s)
            err = abs(Fraction(float(r)) - 1 / Fraction(float(s)))
            assert err <= Fraction(_fp32_ulp(r)) / 2


def test_scale_degenerate_amax_keeps_previous(oracle_mod):
    assert oracle_mod.scale_from_amax(0.0, E4M3, 3.0) == np.float32(3.0)
    assert oracle_mod.scale_from_amax(np.inf, E4M3, 3.0) == np.float32(3.0)
    assert oracle_mod.scale_from_amax(np.nan, E4M3, 3.0) == np.float32(3.0)
    tiny = np.float32(1e-44)  # 448 / tiny overflows fp32
    assert oracle_mod.scale_from_amax(tiny, E4M3, 3.0) == np.finfo(np.float32).max


# --------------------------------------------------------------- history ----

def _const_tensor(amax, n=64):
    v = np.full(n, amax / 2, np.float32)
    v[3] = -amax
    return _bf16_bits(v)


def test_history_spike_golden(oracle_mod):
    from oracle.recipe import DelayedRecipe

    rows = {int(r[0]): (float(r[1]), float(r[2]), int(r[3])) for r in _rows("history_spike.txt")}
    R = DelayedRecipe(1, history_len=16)
    R.set_state(0, [1.0] * 16, 448.0)
    for step in range(40):
        spike = 64.0 if step == 20 else 1.0
        st = R.t[0]
        used = st.scale
        R.quantize(0, _const_tensor(spike), E4M3)
        sat = st.n_saturated
        if step in rows:
            a, want_scale, want_sat = rows[step]
            assert a == spike
            assert float(used) == want_scale, (step, used)
            assert (sat > 0) == bool(want_sat), (step, sat)
        R.update()
    assert len(rows) == 10


def test_history_lag_and_underflow_after_spike(oracle_mod):
    # After the spike the scale is 448/64 = 7, so values 2^-13 (x*7 < 2^-10)
    # that survived before now flush to zero: underflow rises for 16 steps.
    from oracle.recipe import DelayedRecipe

    R = DelayedRecipe(1, history_len=16)
    R.set_state(0, [1.0] * 16, 448.0)
    und = []
    for step in range(40):
        v = np.full(32, 2.0 ** -13, np.float32)
        v[0] = 64.0 if step == 20 else 1.0
        R.quantize(0, _bf16_bits(v), E4M3)
        und.append(R.t[0].n_underflow)
        R.update()
    assert und[:21] == [0] * 21
    assert und[21:37] == [31] * 16
    assert und[37:] == [0] * 3


def test_history_most_recent_rule(oracle_mod):
    from oracle.recipe import ALGO_MOST_RECENT, DelayedRecipe

    R = DelayedRecipe(1, history_len=4, algo=ALGO_MOST_RECENT)
    for a in (2.0, 8.0, 4.0):
        R.quantize(0, _const_tensor(a), E4M3)
        R.update()
        assert float(R.t[0].scale) == 448.0 / a
        assert [float(h) for h in R.t[0].history][-1] == a


def test_history_window_brute_force(oracle_mod):
    from oracle.recipe import DelayedRecipe

    rng = np.random.default_rng(2)
    for H in (1, 2, 3, 16):
        R = DelayedRecipe(1, history_len=H)
        amaxes = [float(np.float32(2.0 ** rng.integers(-6, 8))) for _ in range(3 * H + 5)]
        for t, a in enumerate(amaxes):
            R.quantize(0, _const_tensor(a), E5M2)
            R.update()
            window = amaxes[max(0, t - H + 1): t + 1]
            assert float(R.t[0].scale) == 57344.0 / max(window)


def test_update_only_touches_recorded_tensors(oracle_mod):
    from oracle.recipe import DelayedRecipe

    R = DelayedRecipe(2, history_len=4)
    R.quantize(0, _const_tensor(2.0), E4M3)
    R.update()
    assert float(R.t[0].scale) == 224.0 and float(R.t[1].scale) == 1.0
    assert [float(h) for h in R.t[1].history] == [0.0] * 4


# ------------------------------------------------------------------ GEMM ----

def _dec_fraction(code, fmt, oracle_mod):
    v = oracle_mod.decode(np.array([code], np.uint8), fmt)[0]
    return Fraction(float(v))


@pytest.mark.parametrize("afmt,bfmt", [(E4M3, E4M3), (E5M2, E4M3), (E5M2, E5M2)])
def test_gemm_every_code_pair_exact(oracle_mod, afmt, bfmt):
    a_ok = [c for c in range(256) if np.isfinite(oracle_mod.decode(np.array([c], np.uint8), afmt)[0])]
    b_ok = [c for c in range(256) if np.isfinite(oracle_mod.decode(np.array([c], np.uint8), bfmt)[0])]
    A = np.array(a_ok, np.uint8).reshape(-1, 1)
    B = np.array(b_ok, np.uint8).reshape(-1, 1)
    acc, ab, _ = oracle_mod.gemm(A, afmt, B, bfmt, 1.0, want_bf16=False)
    fa = [_dec_fraction(c, afmt, oracle_mod) for c in a_ok]
    fb = [_dec_fraction(c, bfmt, oracle_mod) for c in b_ok]
    for i in range(len(a_ok)):
        for j in range(len(b_ok)):
            assert Fraction(acc[i, j]) == fa[i] * fb[j]
            assert Fraction(ab[i, j]) == abs(fa[i] * fb[j])


def _nearest_bf16_ok(bits, exact):
    """bits is a nearest bf16 to the rational ``exact`` (ties: even)."""
    def val(b):
        return Fraction(float((np.array([b], np.uint32) << 16).view(np.float32)[0]))
    v = val(bits)
    d = abs(v - exact)
    for nb in ((bits + 1) & 0xFFFF, (bits - 1) & 0xFFFF):
        if (nb & 0x7F80) == 0x7F80:
            continue
        dn = abs(val(nb) - exact)
        if dn < d or (dn == d and (nb & 1) == 0 and (bits & 1) == 1):
            return False
    return True


def test_gemm_random_tiny_exact(oracle_mod):
    rng = np.random.default_rng(4)
    for trial in range(30):
        M, N, K = rng.integers(1, 9, 3)
        afmt, bfmt = rng.integers(0, 2, 2)
        A = rng.integers(0, 256, (M, K)).astype(np.uint8)
        B = rng.integers(0, 256, (N, K)).astype(np.uint8)
        # drop NaN / Inf codes
        A[~np.isfinite(oracle_mod.decode(A, afmt))] = 0x38 if afmt == E4M3 else 0x3C
        B[~np.isfinite(oracle_mod.decode(B, bfmt))] = 0x01
        factor = np.float32(rng.uniform(0.25, 4.0))
        acc, ab, out = oracle_mod.gemm(A, afmt, B, bfmt, factor)
        for m in range(M):
            for n in range(N):
                terms = [_dec_fraction(A[m, k], afmt, oracle_mod) * _dec_fraction(B[n, k], bfmt, oracle_mod)
                         for k in range(K)]
                exact = sum(terms, Fraction(0))
                eabs = sum((abs(t) for t in terms), Fraction(0))
                # products are exact in fp64; the fp64 running sum may round when
                # the terms span more than 53 bits: |err| <= K * 2^-53 * sum|t|
                bound = int(K) * Fraction(1, 2 ** 53) * eabs
                assert abs(Fraction(acc[m, n]) - exact) <= bound, (trial, m, n)
                assert abs(Fraction(ab[m, n]) - eabs) <= bound
                assert _nearest_bf16_ok(int(out[m, n]), Fraction(acc[m, n]) * Fraction(float(factor)))


def test_gemm_identity_weight(oracle_mod):
    rng = np.random.default_rng(8)
    K = 48
    X = rng.integers(0, 0x7E, (5, K)).astype(np.uint8)
    W = np.zeros((K, K), np.uint8)
    np.fill_diagonal(W, 0x38)  # E4M3 1.0
    acc, _, _ = oracle_mod.gemm(X, E4M3, W, E4M3, 1.0, want_bf16=False)
    assert np.array_equal(acc, oracle_mod.decode(X, E4M3))


def test_gemm_single_k_and_orientation(oracle_mod):
    # D[m, n] = A[m, k0] * B[n, k0]: only column k0 nonzero, distinct values
    M, N, K, k0 = 3, 5, 7, 4
    A = np.zeros((M, K), np.uint8)
    B = np.zeros((N, K), np.uint8)
    A[:, k0] = [0x38, 0x40, 0x48]          # 1, 2, 4
    B[:, k0] = [0x38, 0x39, 0x3A, 0x3B, 0xB8]  # 1, 1.125, 1.25, 1.375, -1
    acc, _, _ = oracle_mod.gemm(A, E4M3, B, E4M3, 1.0, want_bf16=False)
    want = np.outer([1, 2, 4], [1, 1.125, 1.25, 1.375, -1])
    assert np.array_equal(acc, want)


def test_gemm_row_subset_matches_full(oracle_mod):
    rng = np.random.default_rng(12)
    A = rng.integers(0, 0x70, (40, 33)).astype(np.uint8)
    B = rng.integers(0, 0x70, (21, 33)).astype(np.uint8)
    full, fab, fout = oracle_mod.gemm(A, E4M3, B, E5M2, 0.5)
    rows = np.array([39, 0, 17, 17, 5])
    sub, sab, sout = oracle_mod.gemm(A, E4M3, B, E5M2, 0.5, rows=rows)
    assert np.array_equal(sub, full[rows]) and np.array_equal(sout, fout[rows])
