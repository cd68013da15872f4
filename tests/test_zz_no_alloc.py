"""fp8_quantize_current_noalloc: the current-scaling cast for callers that
cannot allocate device memory while they run (e.g. code inside a framework
that owns all device memory, or that must not risk an allocation's device-wide
synchronisation).  It keeps its cross-block scratch in a static array inside
the library instead of memory the caller or the library allocates.

The GPU test calls it through the C ABI twice in a row (different sizes and
formats, so the second call reuses scratch the first one left behind) and
checks codes, scale, 1/scale and counts against fp8_amax_quantize in CURRENT
mode on a fresh recipe, bit for bit (the tolerance of every cast test).  This
file is collected last so that a run stopping at the first failure has run
everything else already."""
import numpy as np
import pytest
import torch

from fp8_mixed_precision_history_gb300 import synthetic


def _reference(fp8, x, fmt):
    R = fp8.Recipe(1)
    q = R.quantize(0, x, fmt, fp8.CURRENT)
    st, _ = R.get_state(0)
    R.close()
    return q, st


def _f32(v):
    return int(np.array([v], np.float32).view(np.uint32)[0])


@pytest.mark.gpu
def test_noalloc_matches_current_scaling_cast_twice(gpu_lib):
    fp8 = gpu_lib
    cases = [(3_000_017, 21, fp8.E4M3), (65536 * 3 + 48, 22, fp8.E5M2), (1000, 23, fp8.E4M3)]
    for n, seed, fmt in cases:
        x = synthetic.spiky((n,), seed).cuda()
        out = torch.full((n,), 0xAB, dtype=torch.uint8, device="cuda")
        scale = torch.zeros(2, dtype=torch.float32, device="cuda")
        counts = torch.zeros(2, dtype=torch.int64, device="cuda")
        fp8.fp8_quantize_current_noalloc(x, n, fmt, out, scale, counts)
        torch.cuda.synchronize()
        q_ref, st = _reference(fp8, x, fmt)
        assert torch.equal(out, q_ref), f"codes differ for n={n}"
        s = scale.cpu().numpy()
        assert _f32(s[0]) == _f32(st["cast_scale"]) and _f32(s[1]) == _f32(st["cast_scale_inv"])
        c = counts.cpu().numpy()
        assert int(c[0]) == st["n_saturated"] and int(c[1]) == st["n_underflow"]


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
