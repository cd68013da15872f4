"""bench.py's single-kernel cases and the MX step run on the GPU and print
sane figures (a smoke test of the measurement code, not of the numerics)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIMITS = {"gemm": (500, 5000), "mx_gemm": (300, 5000), "cast": (500, 9000), "cast_t": (500, 9000),
          "mx_quant": (300, 9000), "grad_ar": (300, 12000)}


@pytest.mark.parametrize("case", sorted(LIMITS))
def test_case_runs(gpu_lib, case):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--case", case, "--steps", "2",
                        "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1]
    d = json.loads(line)
    lo, hi = LIMITS[case]
    assert d["case"].split()[0] == case and lo < d["achieved"] < hi, d


def test_mx_step(gpu_lib):
    import torch

    sys.path.insert(0, ROOT)
    import bench

    d = bench.mx_step(gpu_lib, torch.device("cuda", 0), steps=2, warmup=1)
    assert 200 < d["value"] < 5000
    assert set(d["kernel_ms_per_step"]) == {"quant", "gemm"}
    assert d["kernel_ms_per_step"]["gemm"] < d["ms_per_step"]


def test_loop32_reports_every_tensor_every_step(gpu_lib, tmp_path):
    """The 32-step loop at 16384 tokens: one state record per tensor per step,
    and the saturation burst of the spike step in the activations' counts."""
    out = tmp_path / "loop32.jsonl"
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--loop32", str(out)],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    recs = [json.loads(ln) for ln in out.read_text().splitlines()]
    assert d["case"] == "loop32" and d["records"] == len(recs) == 32 * 4 * 4
    assert 500 < d["tflops_median"] < 5000
    sat = d["x_saturated_per_step"]
    assert sat[20] > 1000 * max(1, max(sat[:20]))
    und = d["x_underflow_per_step"]
    assert min(und[21:32]) > 2 * (sum(und[16:20]) / 4)


@pytest.mark.parametrize("transposed", [False, True])
def test_step_line_both_backward_layouts(gpu_lib, transposed):
    """The bench step, short: backward operands read MN-major (default) or from
    transposed copies (the Hopper layout); both print a sane contract line."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3", "--no-cpu-baseline",
           "--no-e2e", "--no-sweep", "--no-mx"] + (["--transposed-copies"] if transposed else [])
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    assert 500 < d["value"] < 5000 and d["gpu_launches"] == 3 * 25
    assert d["config"]["cast_bytes_per_step"] == (4 if transposed else 3) * 738197504
    assert d["roofline"]["bound"] == "tensor" and 0.1 < d["roofline"]["frac"] < 1.5
