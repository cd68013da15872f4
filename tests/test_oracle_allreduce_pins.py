"""Pins for the oracle's FP8 (E5M2) gradient all-reduce with automatic
scaling ("FP8 and low-precision formats", use cases: E5M2 for gradient
communication; FP8-LM forum thread: automatic scaling during the all-reduce).

Pinned by a hand-worked example (tests/golden/allreduce_e5m2_example.txt), by
its reduction to the pinned per-tensor cast for one rank, and by brute force:
exact rational sums with E5M2 rounding found by enumerating every code."""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

E5M2 = oracle.E5M2
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "allreduce_e5m2_example.txt")


def _bits(v):
    a = np.asarray(v, np.float32)
    assert np.all(a.view(np.uint32) & 0xFFFF == 0)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def test_hand_worked_example():
    rows, scale = [], None
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        f = line.split()
        if f[0] == "scale":
            scale = (float(f[1]), float(f[2]))
        else:
            rows.append((float(f[0]), float(f[1]), int(f[2])))
    g = np.stack([_bits([r[0] for r in rows]), _bits([r[1] for r in rows])])
    out, codes, (s, sinv) = oracle.allreduce_e5m2(g)
    assert abs(float(s) - scale[0]) <= scale[1]
    assert list(codes) == [r[2] for r in rows]


def test_scale_rule():
    for a in (1e-3, 0.7, 3.0, 448.0, 1e30):
        # one rank: the per-tensor current scale of an E5M2 cast (pinned)
        assert oracle.allreduce_scale(a, 1) == oracle.scale_from_amax(np.float32(a), E5M2)
    assert oracle.allreduce_scale(0.0, 4) == 1.0
    assert oracle.allreduce_scale(float("inf"), 2) == 1.0
    assert oracle.allreduce_scale(2.0 ** -133, 1) == np.finfo(np.float32).max  # quotient overflows
    # world * amax overflows fp32: clamped to FLT_MAX before the division
    big = np.float32(3.0e38)
    assert oracle.allreduce_scale(big, 4) == np.float32(57344.0) / np.finfo(np.float32).max


@pytest.mark.parametrize("average", [False, True])
def test_one_rank_is_the_per_tensor_round_trip(average):
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(500) * 0.01).astype(np.float32)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    out, codes, (s, sinv) = oracle.allreduce_e5m2(xb[None, :], average=average)
    a = oracle.amax(xb)
    s_ref = oracle.scale_from_amax(a, E5M2)
    q, _, _ = oracle.cast(xb, s_ref, E5M2)
    assert s == s_ref and np.array_equal(codes, q)
    y = (oracle.decode(q, E5M2).astype(np.float32) * np.float32(oracle.reciprocal(s_ref))).astype(np.float32)
    assert np.array_equal(out, oracle.f64_to_bf16(y.astype(np.float64)))


def _e5m2_rne(v):
    """Nearest finite E5M2 value to the exact rational v, ties to an even code,
    saturating: by enumeration of all 123 non-negative finite codes."""
    vals = [(Fraction(float(oracle.decode(np.array([c], np.uint8), E5M2)[0])), c) for c in range(0x7C)]
    mag = abs(v)
    if mag > vals[-1][0]:
        best = vals[-1][1]
    else:
        d = min(abs(mag - x) for x, _ in vals)
        cands = [c for x, c in vals if abs(mag - x) == d]
        best = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
    return best | (0x80 if v < 0 else 0)


@pytest.mark.parametrize("world,average", [(2, False), (3, True), (5, False), (4, True)])
def test_brute_force_small(world, average):
    rng = np.random.default_rng(world * 7 + average)
    n = 40
    mag = np.exp(rng.uniform(np.log(1e-4), np.log(10.0), (world, n)))
    x = (mag * np.where(rng.random((world, n)) < 0.5, -1, 1)).astype(np.float32)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    out, codes, (s, sinv) = oracle.allreduce_e5m2(xb, average=average)
    xv = oracle.bf16_to_f32(xb)
    amax = np.float32(np.max(np.abs(xv)))
    d = np.float32(world) * amax
    s_ref = np.float32(57344.0) / d
    assert s == s_ref
    f = np.float32(np.float32(1.0) / s_ref)
    if average:
        f = np.float32(f / np.float32(world))
    for i in range(n):
        total = Fraction(0)
        for r in range(world):
            p = np.float32(xv[r, i] * s_ref)  # fp32 product
            total += Fraction(float(oracle.decode(np.array([_e5m2_rne(Fraction(float(p)))], np.uint8), E5M2)[0]))
        c = _e5m2_rne(total)
        assert codes[i] == c, (i, codes[i], c)
        y = np.float32(np.float32(oracle.decode(np.array([c], np.uint8), E5M2)[0]) * f)
        assert out[i] == oracle.f64_to_bf16(np.array([float(y)]))[0]
