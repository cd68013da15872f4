"""fp8_quantize_current_noalloc: the current-scaling cast for callers that
cannot allocate device memory while they run (e.g. code inside a framework
that owns all device memory, or that must not risk an allocation's device-wide
synchronisation).  It keeps its cross-block scratch in a static array inside
the library instead of memory the caller or the library allocates.

The GPU tests call it through the C ABI several times in a row (different
sizes and formats, so each call reuses scratch the previous one left behind)
and check codes, scale, 1/scale and counts bit for bit against the oracle's
current-scaling cast and against fp8_amax_quantize in CURRENT mode on a fresh
recipe (the tolerance of every cast test).  Edge cases: an all-zero tensor and
tensors holding Inf or NaN (scale stays 1), and a call without counts followed
by one with counts (the scratch's completion tickets are cleared per call).
This file is collected last so that a run stopping at the first failure has
run everything else already."""
import numpy as np
import pytest
import torch

import oracle
from fp8_mixed_precision_history_gb300 import synthetic


def _reference(fp8, x, fmt):
    R = fp8.Recipe(1)
    q = R.quantize(0, x, fmt, fp8.CURRENT)
    st, _ = R.get_state(0)
    R.close()
    return q, st


def _f32(v):
    return int(np.array([v], np.float32).view(np.uint32)[0])


def _noalloc(fp8, x, fmt, with_counts=True):
    n = x.numel()
    out = torch.full((n,), 0xAB, dtype=torch.uint8, device="cuda")
    scale = torch.zeros(2, dtype=torch.float32, device="cuda")
    counts = torch.full((2,), -1, dtype=torch.int64, device="cuda") if with_counts else None
    fp8.fp8_quantize_current_noalloc(x, n, fmt, out, scale, counts)
    torch.cuda.synchronize()
    return out, scale.cpu().numpy(), None if counts is None else counts.cpu().numpy()


def _nan_code(c, fmt):
    """NaN codes of the format: E4M3 S.1111.111; E5M2 S.11111.{01,10,11}."""
    m = c & 0x7F
    return m == 0x7F if fmt == 0 else m > 0x7C


def _check(fp8, x, fmt, with_counts=True):
    """One allocation-free call against the oracle and against the recipe cast."""
    out, s, c = _noalloc(fp8, x, fmt, with_counts)
    xb = synthetic.bits(x)
    a = oracle.amax(xb)
    os_ = oracle.scale_from_amax(a, fmt, np.float32(1.0))
    oq, ns, nu = oracle.cast(xb, os_, fmt)
    got = synthetic.codes(out)
    nan_in = np.isnan(oracle.bf16_to_f32(xb))
    assert np.array_equal(got[~nan_in], oq[~nan_in]), f"codes differ from the oracle (n={x.numel()})"
    assert _nan_code(got[nan_in], fmt).all(), "a NaN input did not give a NaN code"
    assert _f32(s[0]) == _f32(os_) and _f32(s[1]) == _f32(oracle.reciprocal(os_)), "scale differs from the oracle"
    if c is not None:
        assert int(c[0]) == ns and int(c[1]) == nu, f"counts {c.tolist()} vs oracle {(ns, nu)}"
    q_ref, st = _reference(fp8, x, fmt)
    assert torch.equal(out, q_ref), "codes differ from fp8_amax_quantize CURRENT"
    assert _f32(s[0]) == _f32(st["cast_scale"]) and _f32(s[1]) == _f32(st["cast_scale_inv"])
    if c is not None:
        assert int(c[0]) == st["n_saturated"] and int(c[1]) == st["n_underflow"]


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_recipe_cast_in_a_row(gpu_lib):
    fp8 = gpu_lib
    cases = [(3_000_017, 21, fp8.E4M3), (65536 * 3 + 48, 22, fp8.E5M2), (1000, 23, fp8.E4M3),
             (1, 24, fp8.E5M2), ((1 << 24) + 5, 25, fp8.E5M2)]
    for n, seed, fmt in cases:
        _check(fp8, synthetic.spiky((n,), seed).cuda(), fmt)


@pytest.mark.gpu
def test_noalloc_special_inputs(gpu_lib):
    """All zeros: amax 0, scale stays 1, every code 0.  Inf or NaN anywhere: the
    amax is not finite, so the scale stays 1; Inf saturates (and is counted),
    NaN stays NaN."""
    fp8 = gpu_lib
    n = 70001
    for fmt in (fp8.E4M3, fp8.E5M2):
        _check(fp8, torch.zeros(n, dtype=torch.bfloat16, device="cuda"), fmt)
        for special in (float("inf"), float("-inf"), float("nan")):
            x = synthetic.normal((n,), 1.0, 26)
            x[[5, 40000, n - 1]] = special
            _check(fp8, x.cuda(), fmt)


@pytest.mark.gpu
def test_noalloc_without_counts_then_with(gpu_lib):
    """counts_out = NULL: the cast's last block leaves early.  The next call
    must still count correctly (each call starts its tickets at zero)."""
    fp8 = gpu_lib
    x = synthetic.spiky((900_001,), 27).cuda()
    _check(fp8, x, fp8.E4M3, with_counts=False)
    _check(fp8, x, fp8.E4M3, with_counts=True)
    _check(fp8, synthetic.spiky((123_457,), 28).cuda(), fp8.E5M2, with_counts=False)
    _check(fp8, synthetic.spiky((123_457,), 28).cuda(), fp8.E5M2, with_counts=True)


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_its_scratch(gpu_lib):
    fp8 = gpu_lib
    x = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(64, dtype=torch.uint8, device="cuda")
    scale = torch.empty(2, dtype=torch.float32, device="cuda")
    with pytest.raises(fp8.Fp8Error) as e:
        fp8.fp8_quantize_current_noalloc(x, fp8.NOALLOC_MAX_ELEMENTS + 1, fp8.E4M3, out, scale)
    assert e.value.status == 1 and "scratch" in str(e.value)


def test_noalloc_limit_matches_header():
    import os
    import re

    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "include", "fp8lin.h")).read()
    m = re.search(r"#define FP8_NOALLOC_MAX_ELEMENTS \(\(int64_t\)1 << (\d+)\)", hdr)
    import fp8_mixed_precision_history_gb300 as fp8

    assert m and fp8.NOALLOC_MAX_ELEMENTS == 1 << int(m.group(1))
