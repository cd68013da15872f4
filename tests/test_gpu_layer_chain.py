"""The transformer layer's step with its GEMMs chained through their epilogues
("4.2 Hopper I -- Transformer Engine / FP8", S4.2.4: the FP32 result is
multiplied by 1/scale "or composed with the next stage's scale"; S4.2.6: the
te.TransformerLayer with HYBRID delayed scaling, history 16, "max").

Per step, as the benchmark's chained step runs it: QKV's forward writes E4M3
codes (its output tensor's delayed scale); FC1's forward applies GELU and
writes FC2's E4M3 operand and the bf16 derivative gelu'(y); FC2's dgrad
multiplies by that derivative and writes FC1's E5M2 output gradient; the other casts come from bf16
inputs; then one scale update.  The oracle recipe follows every tensor:

* every cast from bf16: codes and state bit for bit (oracle.DelayedRecipe);
* every epilogue cast: its codes equal the oracle's cast of the kernel's fp32
  values (the same GEMM with an fp32 output), bit for bit, and the oracle
  records that cast's amax and counts itself (record_cast);
* every fp32 value of an epilogue output against the oracle's fp64 chain on
  sampled rows (exact sums, GELU and gelu' in fp64) within the propagated
  bound, and the saved derivative against gelu'(y);
* the GEMMs that consume epilogue codes against the oracle's GEMM of those
  codes with the recorded 1/scale, on sampled rows, within the accumulation
  bound for any operand distribution (gpu_util.fp32_mma_rel);
* after each update, every tensor's scale, 1/scale, history and counts.
At reduced size over 6 steps; at full size (8192 tokens, hidden 4096, FFN
16384) over 2 steps.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.recipe import DelayedRecipe
from fp8_mixed_precision_history_gb300 import synthetic
from gpu_util import check_gemm_sample, check_state, fp32_mma_rel, to_host_u16, to_host_u8
from test_gpu_gemm_act import _act_bound, _aux_bound

pytestmark = pytest.mark.gpu


def _layers(full):
    if full:
        return synthetic.TE_LAYERS
    return (("qkv", 128, 384), ("proj", 128, 128), ("fc1", 128, 512), ("fc2", 512, 128))


class Chain:
    """The chained step through the C ABI (the GPU side of the test)."""

    def __init__(self, fp8, layers, T, dev):
        self.fp8, self.T, self.dev = fp8, T, dev
        self.L = {n: (fin, fout) for n, fin, fout in layers}
        self.names = [n for n, _, _ in layers]
        self.id = {n: 4 * i for i, n in enumerate(self.names)}
        self.R = fp8.Recipe(4 * len(layers))
        u8 = dict(dtype=torch.uint8, device=dev)
        self.w = {n: synthetic.normal((fo, fi), 0.02, synthetic.seed_for(6, i, "w"), device=dev)
                  for i, (n, fi, fo) in enumerate(layers)}
        self.wq = {n: torch.empty((fo, fi), **u8) for n, (fi, fo) in self.L.items()}
        self.xq = {n: torch.empty((T, fi), **u8) for n, (fi, fo) in self.L.items()}
        self.dq = {n: torch.empty((T, fo), **u8) for n, (fi, fo) in self.L.items()}
        self.yq = torch.empty((T, self.L["qkv"][1]), **u8)
        self.h = torch.empty((T, self.L["fc1"][1]), dtype=torch.bfloat16, device=dev)

    def x(self, n, step):
        i = self.names.index(n)
        return synthetic.normal((self.T, self.L[n][0]), 1.0 * 1.03 ** step, synthetic.seed_for(6, i, "x", step),
                                device=self.dev)

    def dy(self, n, step):
        i = self.names.index(n)
        return synthetic.grad_like((self.T, self.L[n][1]), synthetic.seed_for(6, i, "dy", step), device=self.dev)


def _cast_check(C, OR, tid, t, q, fmt, what):
    oq = OR.quantize(tid, synthetic.bits(t), fmt)
    assert np.array_equal(to_host_u8(q), oq), f"{what}: codes differ from the oracle"
    check_state(C.R, OR, tid, what)


def _epilogue_check(C, OR, tid, q, v32, fmt, what):
    """Codes of an epilogue cast == the oracle's cast of the kernel's fp32
    values with the tensor's delayed scale; the oracle records the cast."""
    vh = v32.cpu().numpy()
    oq, ns, nu, am = oracle.cast_f32(vh, OR.t[tid].scale, fmt)
    bad = np.flatnonzero(to_host_u8(q).ravel() != oq.ravel())
    assert bad.size == 0, f"{what}: {bad.size} epilogue codes differ, first {bad[:4]}"
    OR.record_cast(tid, am, ns, nu, fmt)
    check_state(C.R, OR, tid, what)
    return vh


def _rows(T, full):
    return np.sort(np.random.default_rng(T).choice(T, 48 if full else T, replace=False))


def _run_chain(fp8, full, steps):
    layers = _layers(full)
    T = 8192 if full else 256
    dev = torch.device("cuda")
    C = Chain(fp8, layers, T, dev)
    R, fp = C.R, fp8
    OR = DelayedRecipe(4 * len(layers))
    idd = C.id
    rows = _rows(T, full)
    E4, E5 = fp8.E4M3, fp8.E5M2
    # warm start: current-scaling casts of step 0's bf16 inputs, then an update
    for n in C.names:
        for tid, t, fmt in ((idd[n], C.x(n, 0) if n != "fc2" else None, 0), (idd[n] + 1, C.w[n], 0),
                            (idd[n] + 2, C.dy(n, 0) if n != "fc1" else None, 1)):
            if t is None:
                continue
            R.quantize(tid, t, fmt, fp.CURRENT)
            OR.quantize(tid, synthetic.bits(t), fmt, current=True)
    R.update_scales()
    OR.update()
    for step in range(steps):
        f32 = {}
        # ---------------- forward
        for n in C.names:
            i = idd[n]
            if n != "fc2":
                x = C.x(n, step)
                R.quantize(i, x, E4, out=C.xq[n])
                _cast_check(C, OR, i, x, C.xq[n], 0, f"step {step} {n} X")
            R.quantize(i + 1, C.w[n], E4, out=C.wq[n])
            _cast_check(C, OR, i + 1, C.w[n], C.wq[n], 0, f"step {step} {n} W")
            fac = np.float32(OR.t[i].cast_scale_inv) * np.float32(OR.t[i + 1].cast_scale_inv)
            if n == "qkv":
                R.gemm(i, C.xq[n], E4, i + 1, C.wq[n], E4, out_dtype=fp.OUT_E4M3, out=C.yq, amax_out_id=i + 3)
                y32 = R.gemm(i, C.xq[n], E4, i + 1, C.wq[n], E4, out_dtype=fp.OUT_F32)
                torch.cuda.synchronize()
                vh = _epilogue_check(C, OR, i + 3, C.yq, y32, 0, f"step {step} qkv output codes")
                acc, absacc, _ = oracle.gemm(to_host_u8(C.xq[n]), 0, to_host_u8(C.wq[n]), 0, fac, rows=rows,
                                             want_bf16=False)
                assert np.all(np.abs(vh[rows] - acc * float(fac)) <= 1e-6 * absacc * float(fac))
            elif n == "fc1":
                R.gemm(i, C.xq[n], E4, i + 1, C.wq[n], E4, out_dtype=fp.OUT_E4M3, out=C.xq["fc2"],
                       amax_out_id=idd["fc2"], act=fp.ACT_GELU, aux=C.h)
                v32 = R.gemm(i, C.xq[n], E4, i + 1, C.wq[n], E4, out_dtype=fp.OUT_F32, act=fp.ACT_GELU)
                torch.cuda.synchronize()
                vh = _epilogue_check(C, OR, idd["fc2"], C.xq["fc2"], v32, 0, f"step {step} fc1 -> fc2 X codes")
                acc, absacc, _ = oracle.gemm(to_host_u8(C.xq[n]), 0, to_host_u8(C.wq[n]), 0, fac, rows=rows,
                                             want_bf16=False)
                y64 = acc * float(fac)
                bound_y = 1e-6 * absacc * float(fac)
                bound = _act_bound(y64, bound_y, fp.ACT_GELU)
                assert np.all(np.abs(vh[rows] - oracle.gelu(y64)) <= bound), f"step {step} fc1 gelu values"
                f32["h"] = to_host_u16(C.h)
                dg = oracle.bf16_to_f32(f32["h"][rows]).astype(np.float64)
                assert np.all(np.abs(dg - oracle.dgelu(y64)) <= _aux_bound(y64, bound_y)), f"step {step} gelu'"
            else:
                y = R.gemm(i, C.xq[n], E4, i + 1, C.wq[n], E4, amax_out_id=i + 3)
                yb = to_host_u16(y)
                OR.record_amax(i + 3, np.max(np.abs(oracle.bf16_to_f32(yb))))
                check_state(R, OR, i + 3, f"step {step} {n} output amax")
                if n == "fc2":  # consumes the epilogue codes with their recorded 1/scale
                    check_gemm_sample(None, y, to_host_u8(C.xq[n]), 0, to_host_u8(C.wq[n]), 0, fac, rows,
                                      rel=fp32_mma_rel(C.L[n][0]))
        # ---------------- backward
        for n in reversed(C.names):
            i = idd[n]
            if n != "fc1":
                dy = C.dy(n, step)
                R.quantize(i + 2, dy, E5, out=C.dq[n])
                _cast_check(C, OR, i + 2, dy, C.dq[n], 1, f"step {step} {n} dY")
            fac = np.float32(OR.t[i + 2].cast_scale_inv) * np.float32(OR.t[i + 1].cast_scale_inv)
            wT = np.ascontiguousarray(to_host_u8(C.wq[n]).T)
            if n == "fc2":
                R.gemm(i + 2, C.dq[n], E5, i + 1, C.wq[n], E4, out_dtype=fp.OUT_E5M2, out=C.dq["fc1"],
                       amax_out_id=idd["fc1"] + 2, b_major=fp.MN_MAJOR, act=fp.ACT_DGELU, aux=C.h)
                v32 = R.gemm(i + 2, C.dq[n], E5, i + 1, C.wq[n], E4, out_dtype=fp.OUT_F32, b_major=fp.MN_MAJOR,
                             act=fp.ACT_DGELU, aux=C.h)
                torch.cuda.synchronize()
                vh = _epilogue_check(C, OR, idd["fc1"] + 2, C.dq["fc1"], v32, 1, f"step {step} fc2 -> fc1 dY codes")
                acc, absacc, _ = oracle.gemm(to_host_u8(C.dq[n]), 1, wT, 0, fac, rows=rows, want_bf16=False)
                y64 = acc * float(fac)
                gv = oracle.bf16_to_f32(f32["h"][rows]).astype(np.float64)
                bound = _act_bound(y64, 1e-6 * absacc * float(fac), fp.ACT_DGELU, gv)
                assert np.all(np.abs(vh[rows] - y64 * gv) <= bound), f"step {step} fc2 y * gelu' values"
            else:  # dgrad, bf16 out; for fc1 it reads the epilogue's E5M2 codes
                dx = R.gemm(i + 2, C.dq[n], E5, i + 1, C.wq[n], E4, b_major=fp.MN_MAJOR)
                if n == "fc1":
                    check_gemm_sample(None, dx, to_host_u8(C.dq[n]), 1, wT, 0, fac, rows,
                                      rel=fp32_mma_rel(C.L[n][1]))
            dw = R.gemm(i + 2, C.dq[n], E5, i, C.xq[n], E4, a_major=fp.MN_MAJOR, b_major=fp.MN_MAJOR)
            if n in ("fc1", "fc2"):  # wgrad on epilogue codes (fc1: dY; fc2: X)
                fw = np.float32(OR.t[i + 2].cast_scale_inv) * np.float32(OR.t[i].cast_scale_inv)
                wrows = np.sort(np.random.default_rng(step).choice(dw.shape[0], 32, replace=False))
                check_gemm_sample(None, dw, np.ascontiguousarray(to_host_u8(C.dq[n]).T), 1,
                                  np.ascontiguousarray(to_host_u8(C.xq[n]).T), 0, fw, wrows, rel=fp32_mma_rel(T))
            del dw
        R.update_scales()
        OR.update()
        for tid in range(4 * len(C.names)):
            check_state(R, OR, tid, f"step {step} tensor {tid} after update")
    R.check_device_error()
    R.close()


def test_layer_chain_reduced_size(gpu_lib):
    _run_chain(gpu_lib, full=False, steps=6)


def test_layer_chain_full_size(gpu_lib):
    _run_chain(gpu_lib, full=True, steps=2)
