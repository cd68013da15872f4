"""Benchmark: one training step of the per-tensor scaled FP8 linear path.

A step is the whole hot path over the four linear layers of a transformer
layer (hidden 4096, FFN 16384; QKV 4096->12288, proj 4096->4096,
FC1 4096->16384, FC2 16384->4096) at 8192 tokens, HYBRID delayed scaling
with a 16-entry "max" amax history:
  per layer: cast X (E4M3) and W (E4M3), forward GEMM Y = X W^T (output amax
  fused into the epilogue), cast dY (E5M2), dgrad dX = dY W, wgrad
  dW = dY^T X; then one scale update.  The backward GEMMs read the forward
  casts' codes as MN-major operands (W for dgrad, dY and X for wgrad), so no
  cast writes a transposed copy; --transposed-copies runs the layout of the
  Hopper recipe instead (every cast also writes its transpose and all GEMM
  operands are K-major).
The GEMMs do 9895.6 GFLOP per step.

Prints one JSON line.  `value` is step throughput in TFLOP/s with inputs
resident in HBM; `e2e` repeats the measurement through the same C-ABI calls
with the step's inputs copied from pinned host memory and its outputs copied
back inside the timed region.  `--impl reference` times the CPU oracle on a
bounded sample of the same step instead.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

TOKENS = 8192
METRIC = "FP8 scaled-GEMM TFLOP/s and amax+cast GB/s at 1 GB300, % of roofline"
WORKLOAD = "te_layer_fwd_dgrad_wgrad_tokens8192"


def layers():
    from fp8_mixed_precision_history_gb300 import synthetic

    return synthetic.TE_LAYERS


def step_flops(T=TOKENS):
    return sum(3 * 2 * T * fin * fout for _, fin, fout in layers())


def cast_bytes(T=TOKENS, transposed=False):
    """Algorithmic bytes of the step's casts: 2 B read + 1 B q per element, and
    1 B more for q^T with transposed copies."""
    n = sum(T * fin + fout * fin + T * fout for _, fin, fout in layers())
    return (4 if transposed else 3) * n


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# Dense FP8 tensor-core work per SM per clock: 2 x the 8192 bf16 FLOP of a
# 5th-generation tensor core (152 SMs x 16384 x 1.807 GHz = the 4.5 PFLOP/s
# dense FP8 figure quoted for the part).
FP8_FLOP_PER_SM_CLOCK = 16384
# A timed region shorter than this runs at the burst clocks: its GEMMs are held
# to the burst peak; longer regions to the sustained (power-capped) one.
BURST_REGION_S = 1.0


def fp8_peaks(peaks, src, region_s, sm_mhz, num_sms):
    """Dense FP8 denominators of a GEMM figure.  Returns (peak TFLOP/s the frac
    uses, its source, per-clock nominal TFLOP/s at the sampled SM clock or
    None).  The measured peaks are 2 x cuBLAS bf16 (the nominal fp8:bf16
    ratio): burst for a region under BURST_REGION_S, else sustained."""
    if region_s < BURST_REGION_S:
        peak = 2.0 * peaks["bf16_tflops"]
        how = f"2 x bf16_tflops, burst ({src}): timed region {region_s:.2f} s < {BURST_REGION_S:g} s"
    else:
        peak = 2.0 * peaks["bf16_tflops_sustained"]
        how = f"2 x bf16_tflops_sustained ({src}): timed region {region_s:.2f} s"
    clock = None
    if sm_mhz:
        clock = num_sms * FP8_FLOP_PER_SM_CLOCK * sm_mhz * 1e6 / 1e12
    return peak, how, clock


GEMM_PROFILE = os.path.join(ROOT, "profiles", "fp8_gemm_pair_kernel_traffic_te_layer_step_tokens8192.md")
GEMM_SOURCES = ("gemm_tcgen05.cu", "tc_ptx.cuh")


def gemm_source_sha256():
    import hashlib

    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "fp8_mixed_precision_history_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def gemm_traffic():
    """DRAM bytes per GEMM launch of the step (read + write, mean over the
    step's 12 launches) from the committed ncu summary, or None when the
    summary was taken on other kernel sources than the ones built here."""
    import re

    try:
        text = open(GEMM_PROFILE).read()
    except OSError:
        return None
    t = re.search(r"^gemm_traffic_bytes_per_launch: (\d+)$", text, re.M)
    h = re.search(r"^gemm_source_sha256: ([0-9a-f]{64})$", text, re.M)
    if not t or not h or h.group(1) != gemm_source_sha256():
        return None
    return int(t.group(1))


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.idx = device_index
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix=f"fp8lin_clocks_dev{self.idx}_", suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.idx)], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        samples = open(self.path).read().splitlines()
        os.unlink(self.path)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- our arm --

class Step:
    """Device buffers and the launch sequence of one step."""

    def __init__(self, fp8, device, T=TOKENS, seed_base=7000, transposed=False):
        from fp8_mixed_precision_history_gb300 import synthetic

        self.fp8 = fp8
        self.T = T
        self.transposed = transposed
        L = layers()
        # tensor ids: per layer x, w, dy, y
        self.R = fp8.Recipe(4 * len(L), amax_history_len=16)
        self.x, self.w, self.dy = [], [], []
        self.xq, self.xt, self.wq, self.wt, self.dq, self.dt = [], [], [], [], [], []
        self.y, self.dx, self.dw = [], [], []
        u8 = dict(dtype=torch.uint8, device=device)
        bf = dict(dtype=torch.bfloat16, device=device)
        for li, (_, fin, fout) in enumerate(L):
            self.x.append(synthetic.normal((T, fin), 1.0, seed_base + 10 * li, device=device))
            self.w.append(synthetic.normal((fout, fin), 0.02, seed_base + 10 * li + 1, device=device))
            self.dy.append(synthetic.grad_like((T, fout), seed_base + 10 * li + 2, device=device))
            self.xq.append(torch.empty((T, fin), **u8))
            self.wq.append(torch.empty((fout, fin), **u8))
            self.dq.append(torch.empty((T, fout), **u8))
            self.xt.append(torch.empty((fin, T), **u8) if transposed else None)
            self.wt.append(torch.empty((fin, fout), **u8) if transposed else None)
            self.dt.append(torch.empty((fout, T), **u8) if transposed else None)
            self.y.append(torch.empty((T, fout), **bf))
            self.dx.append(torch.empty((T, fin), **bf))
            self.dw.append(torch.empty((fout, fin), **bf))
        # warm start: one current-scaling cast per tensor, then a scale update
        s = torch.cuda.current_stream()
        for li in range(len(L)):
            self._casts(li, fp8.CURRENT, s)
        self.R.update_scales(s)
        torch.cuda.synchronize()
        self.R.check_device_error()

    def _casts(self, li, mode, s, which=("x", "w", "dy")):
        fp8, R = self.fp8, self.R
        T = self.T
        if "x" in which:
            x = self.x[li]
            fp8.fp8_amax_quantize(R.handle, 4 * li, x, T, x.shape[1], fp8.E4M3, mode, 0,
                                  self.xq[li], self.xt[li], s)
        if "w" in which:
            w = self.w[li]
            fp8.fp8_amax_quantize(R.handle, 4 * li + 1, w, w.shape[0], w.shape[1], fp8.E4M3, mode, 0,
                                  self.wq[li], self.wt[li], s)
        if "dy" in which:
            dy = self.dy[li]
            fp8.fp8_amax_quantize(R.handle, 4 * li + 2, dy, T, dy.shape[1], fp8.E5M2, mode, 0,
                                  self.dq[li], self.dt[li], s)

    def _gemm(self, a_id, A, adt, a_mn, b_id, B, bdt, b_mn, D, amax_id, s):
        """D = A B^T; an operand stored MN-major (a_mn / b_mn) is [K, M] / [K, N]."""
        fp8 = self.fp8
        M, K = (A.shape[1], A.shape[0]) if a_mn else (A.shape[0], A.shape[1])
        N = B.shape[1] if b_mn else B.shape[0]
        fp8.fp8_gemm_layout(self.R.handle, a_id, A, adt, int(a_mn), A.stride(0), b_id, B, bdt, int(b_mn),
                            B.stride(0), M, N, K, D, fp8.OUT_BF16, D.stride(0), amax_id, s)

    def forward(self, li, s):
        """Y = X W^T, the output's amax recorded for tensor 4*li+3."""
        fp8 = self.fp8
        self._gemm(4 * li, self.xq[li], fp8.E4M3, False, 4 * li + 1, self.wq[li], fp8.E4M3, False,
                   self.y[li], 4 * li + 3, s)

    def dgrad(self, li, s):
        """dX = dY W: B = W^T, i.e. W's codes [out, in] read MN-major."""
        fp8 = self.fp8
        if self.transposed:
            B, b_mn = self.wt[li], False
        else:
            B, b_mn = self.wq[li], True
        self._gemm(4 * li + 2, self.dq[li], fp8.E5M2, False, 4 * li + 1, B, fp8.E4M3, b_mn, self.dx[li], -1, s)

    def wgrad(self, li, s):
        """dW = dY^T X: A = dY^T and B = X^T, i.e. the codes [T, out] and
        [T, in] read MN-major."""
        fp8 = self.fp8
        if self.transposed:
            A, B, mn = self.dt[li], self.xt[li], False
        else:
            A, B, mn = self.dq[li], self.xq[li], True
        self._gemm(4 * li + 2, A, fp8.E5M2, mn, 4 * li, B, fp8.E4M3, mn, self.dw[li], -1, s)

    def launches_per_step(self):
        return 3 * len(self.x) + 3 * len(self.x) + 1

    def run(self, s, ev=None):
        """Enqueue one step on stream s.  ev: optional dict collecting
        (start, end) CUDA events per kernel kind."""
        fp8 = self.fp8

        def timed(kind, fn):
            if ev is None:
                fn()
                return
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(s)
            fn()
            b.record(s)
            ev.setdefault(kind, []).append((a, b))

        for li in range(len(self.x)):
            timed("cast", lambda: self._casts(li, fp8.DELAYED, s, ("x", "w")))
            timed("gemm", lambda: self.forward(li, s))
        for li in reversed(range(len(self.x))):
            timed("cast", lambda: self._casts(li, fp8.DELAYED, s, ("dy",)))
            timed("gemm", lambda: self.dgrad(li, s))
            timed("gemm", lambda: self.wgrad(li, s))
        timed("update", lambda: self.R.update_scales(s))


class ChainedStep:
    """The transformer layer's step with the GEMMs chained through their
    epilogues (the result's 1/scale "composed with the next stage's scale"):
      forward   QKV writes its output as E4M3 codes (the operand of an FP8
                attention, outside this path); proj as bf16 (residual);
                FC1 applies GELU and writes FC2's E4M3 operand, plus the bf16
                derivative gelu'(y) for the backward; FC2 as bf16 (residual)
      backward  FC2's dgrad applies GELU' and writes FC1's E5M2 output
                gradient; FC1's dgrad and wgrad read those codes
    So FC2's X and FC1's dY are never cast from bf16: the step casts X of QKV,
    proj and FC1, the four weights, and dY of FC2, proj and QKV (inputs the
    layer's other operations -- layer norms, attention, residual -- would give
    in bf16).  Every FP8 epilogue output records its amax and counts into its
    tensor's history, like a delayed cast."""

    def __init__(self, fp8, device, T=TOKENS, seed_base=7000):
        from fp8_mixed_precision_history_gb300 import synthetic

        self.fp8 = fp8
        self.T = T
        L = layers()
        self.names = [n for n, _, _ in L]
        self.li = {n: i for i, n in enumerate(self.names)}
        self.R = fp8.Recipe(4 * len(L), amax_history_len=16)
        u8 = dict(dtype=torch.uint8, device=device)
        bf = dict(dtype=torch.bfloat16, device=device)
        self.x, self.w, self.dy = {}, {}, {}
        self.xq, self.wq, self.dq = {}, {}, {}
        self.y, self.dx, self.dw = {}, {}, {}
        for li, (n, fin, fout) in enumerate(L):
            self.w[n] = synthetic.normal((fout, fin), 0.02, seed_base + 10 * li + 1, device=device)
            self.wq[n] = torch.empty((fout, fin), **u8)
            self.xq[n] = torch.empty((T, fin), **u8)
            self.dq[n] = torch.empty((T, fout), **u8)
            self.dw[n] = torch.empty((fout, fin), **bf)
            if n != "fc2":
                self.x[n] = synthetic.normal((T, fin), 1.0, seed_base + 10 * li, device=device)
            if n != "fc1":
                self.dy[n] = synthetic.grad_like((T, fout), seed_base + 10 * li + 2, device=device)
            if n != "fc2":
                self.dx[n] = torch.empty((T, fin), **bf)
            if n in ("proj", "fc2"):
                self.y[n] = torch.empty((T, fout), **bf)
        self.yq_qkv = torch.empty((T, L[self.li["qkv"]][2]), **u8)
        self.h_fc1 = torch.empty((T, L[self.li["fc1"]][2]), **bf)  # gelu' of FC1's output
        # warm start: current-scaling casts of the bf16 inputs, then one step
        # so that the epilogue-cast tensors have a history too
        s = torch.cuda.current_stream()
        for n in self.names:
            i = self.li[n]
            if n in self.x:
                fp8.fp8_amax_quantize(self.R.handle, 4 * i, self.x[n], T, self.x[n].shape[1], fp8.E4M3,
                                      fp8.CURRENT, 0, self.xq[n], None, s)
            fp8.fp8_amax_quantize(self.R.handle, 4 * i + 1, self.w[n], self.w[n].shape[0], self.w[n].shape[1],
                                  fp8.E4M3, fp8.CURRENT, 0, self.wq[n], None, s)
            if n in self.dy:
                fp8.fp8_amax_quantize(self.R.handle, 4 * i + 2, self.dy[n], T, self.dy[n].shape[1], fp8.E5M2,
                                      fp8.CURRENT, 0, self.dq[n], None, s)
        self.R.update_scales(s)
        self.run(s)
        torch.cuda.synchronize()
        self.R.check_device_error()

    def _cast(self, tid, x, dt, out, s):
        self.fp8.fp8_amax_quantize(self.R.handle, tid, x, x.shape[0], x.shape[1], dt, self.fp8.DELAYED, 0, out,
                                   None, s)

    def _gemm(self, a_id, A, adt, a_mn, b_id, B, bdt, b_mn, D, d_dtype, amax_id, s, act=0, aux=None):
        fp8 = self.fp8
        M, K = (A.shape[1], A.shape[0]) if a_mn else (A.shape[0], A.shape[1])
        N = B.shape[1] if b_mn else B.shape[0]
        fp8.fp8_gemm_act(self.R.handle, a_id, A, adt, int(a_mn), A.stride(0), b_id, B, bdt, int(b_mn),
                         B.stride(0), M, N, K, D, d_dtype, D.stride(0), amax_id, act, aux,
                         0 if aux is None else aux.stride(0), s)

    def run(self, s, ev=None):
        fp8 = self.fp8
        E4, E5 = fp8.E4M3, fp8.E5M2

        def timed(kind, fn):
            if ev is None:
                fn()
                return
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(s)
            fn()
            b.record(s)
            ev.setdefault(kind, []).append((a, b))

        ids = {n: 4 * self.li[n] for n in self.names}  # x, w, dy, y = +0, +1, +2, +3
        xq, wq, dq = self.xq, self.wq, self.dq
        # ---- forward
        for n in self.names:
            if n in self.x:
                timed("cast", lambda: self._cast(ids[n], self.x[n], E4, xq[n], s))
            timed("cast", lambda: self._cast(ids[n] + 1, self.w[n], E4, wq[n], s))
            if n == "qkv":
                timed("gemm", lambda: self._gemm(ids[n], xq[n], E4, False, ids[n] + 1, wq[n], E4, False,
                                                 self.yq_qkv, fp8.OUT_E4M3, ids[n] + 3, s))
            elif n == "fc1":  # gelu(y) as FC2's operand; y kept for the backward
                timed("gemm", lambda: self._gemm(ids[n], xq[n], E4, False, ids[n] + 1, wq[n], E4, False,
                                                 xq["fc2"], fp8.OUT_E4M3, ids["fc2"], s, fp8.ACT_GELU,
                                                 self.h_fc1))
            else:
                timed("gemm", lambda: self._gemm(ids[n], xq[n], E4, False, ids[n] + 1, wq[n], E4, False,
                                                 self.y[n], fp8.OUT_BF16, ids[n] + 3, s))
        # ---- backward
        for n in reversed(self.names):
            if n in self.dy:
                timed("cast", lambda: self._cast(ids[n] + 2, self.dy[n], E5, dq[n], s))
            if n == "fc2":  # dY . W through GELU' as FC1's output gradient
                timed("gemm", lambda: self._gemm(ids[n] + 2, dq[n], E5, False, ids[n] + 1, wq[n], E4, True,
                                                 dq["fc1"], fp8.OUT_E5M2, ids["fc1"] + 2, s, fp8.ACT_DGELU,
                                                 self.h_fc1))
            else:
                timed("gemm", lambda: self._gemm(ids[n] + 2, dq[n], E5, False, ids[n] + 1, wq[n], E4, True,
                                                 self.dx[n], fp8.OUT_BF16, -1, s))
            timed("gemm", lambda: self._gemm(ids[n] + 2, dq[n], E5, True, ids[n], xq[n], E4, True,
                                             self.dw[n], fp8.OUT_BF16, -1, s))
        timed("update", lambda: self.R.update_scales(s))

    def launches_per_step(self):
        return len(self.x) + len(self.w) + len(self.dy) + 3 * len(self.names) + 1

    def cast_bytes(self):
        """3 B per element (bf16 read, codes written) of the tensors cast from bf16."""
        return 3 * sum(t.numel() for d in (self.x, self.w, self.dy) for t in d.values())


def chained_bytes(T=TOKENS):
    """Algorithmic HBM bytes per step: (plain step, chained step).  Plain: the
    casts (3 B/element) of X, W, dY of every layer and the GEMMs' FP8 operands
    and bf16 outputs.  Chained: no casts of FC2's X and FC1's dY; QKV's forward
    writes 1 B codes instead of 2 B; FC1's forward writes 1 B codes and the 2 B
    derivative gelu'(y); FC2's dgrad reads the 2 B derivative and writes 1 B
    codes."""
    L = {n: (fin, fout) for n, fin, fout in layers()}
    plain = cast_bytes() + sum(gemm_algorithmic_bytes(T))
    chained = plain - 3 * T * L["fc2"][0] - 3 * T * L["fc1"][1]
    chained -= T * L["qkv"][1]                    # QKV: E4M3 codes instead of bf16
    chained += T * L["fc1"][1] * (1 + 2 - 2)      # FC1: codes + derivative instead of bf16
    chained += T * L["fc2"][0] * (2 + 1 - 2)      # FC2 dgrad: reads aux, writes codes instead of bf16
    return plain, chained


def layer_step(fp8, device, steps=30, warmup=3, plain_ms=None):
    """Times the chained step like the plain step: the steps alone, then a
    second pass with events around each kernel kind for the split."""
    s = torch.cuda.current_stream()
    st = ChainedStep(fp8, device)
    for _ in range(warmup):
        st.run(s)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s)
    for _ in range(steps):
        st.run(s)
    t1.record(s)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    kms, _ = kernel_windows(st, s, steps)
    st.R.check_device_error()
    split = {k: round(v / steps, 4) for k, v in kms.items()}
    plain_b, chained_b = chained_bytes()
    out = {"value": round(step_flops() / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
           "steps": steps, "kernel_ms_per_step": split, "launches_per_step": st.launches_per_step(),
           "cast_bytes_per_step": st.cast_bytes(), "algorithmic_bytes_per_step": chained_b,
           "bytes_saved_vs_plain_step": plain_b - chained_b,
           "gemm_tflops": round(step_flops() / (split["gemm"] * 1e-3) / 1e12, 1),
           "cast_gbs": round(st.cast_bytes() / (split["cast"] * 1e-3) / 1e9, 1),
           "what": "QKV -> E4M3 codes, FC1 -> GELU -> FC2's E4M3 codes (+ bf16 gelu'), "
                   "FC2 dgrad x gelu' -> FC1's E5M2 gradient codes; same layers, tokens and FLOPs"}
    if plain_ms is not None:
        out["ms_saved_vs_plain_step"] = round(plain_ms - ms, 4)
    st.R.close()
    return out


def kernel_windows(step, s, steps):
    """Per-kernel-kind device time over `steps` steps: an event pair around
    each kernel kind on the launching stream.  The events sit between the
    launches, so they also stop each kernel from starting early behind the
    previous one; the step itself is timed without them.  Returns (ms per
    kind summed over the steps, the pass's total ms)."""
    ev = {}
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s)
    for _ in range(steps):
        step.run(s, ev)
    t1.record(s)
    torch.cuda.synchronize()
    return {k: sum(a.elapsed_time(b) for a, b in v) for k, v in ev.items()}, t0.elapsed_time(t1)


def gemm_algorithmic_bytes(T=TOKENS):
    """Operand + output bytes of the step's GEMMs: FP8 A and B read once,
    bf16 D written once (fprop, dgrad, wgrad of every layer)."""
    out = []
    for _, fin, fout in layers():
        for M, N, K in ((T, fout, fin), (T, fin, fout), (fout, fin, T)):
            out.append(M * K + N * K + 2 * M * N)
    return out


def run_ours(args):
    import torch.distributed as dist

    import fp8_mixed_precision_history_gb300 as fp8

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    fp8.load()
    step = Step(fp8, device, seed_base=7000 + 100 * rank, transposed=args.transposed_copies)
    s = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step.run(s)
    torch.cuda.synchronize()

    # ---- device-resident timed region --------------------------------
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s)
    for _ in range(args.steps):
        step.run(s)
    t1.record(s)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms = t0.elapsed_time(t1)
    # per-kernel windows: the same steps again, with an event pair around each
    # kernel kind (those events separate the launches, so this pass is slower
    # and is not the step time)
    kernel_ms, ms_events = kernel_windows(step, s, args.steps)
    clk = clocks.stop()
    step.R.check_device_error()

    peaks, src = load_peaks()
    num_sms = torch.cuda.get_device_properties(device).multi_processor_count
    # ---- FC2 forward alone, the 8192 x 4096 x 16384 shape -------------
    fc2 = gemm_fc2(step, s, local, peaks, src, num_sms)
    # ---- end to end through host buffers -----------------------------
    e2e = None if args.no_e2e else run_e2e(step, s, args)
    sweep = None if args.no_sweep else cast_sweep(fp8, device, peaks["hbm_gbs"])
    mx = None if args.no_mx else mx_step(fp8, device)
    chained = None if args.no_chain else layer_step(fp8, device, plain_ms=ms / args.steps)

    ms_max, value = aggregate(ms, step_flops() * args.steps, world, device)

    fp8_peak, peak_how, clock_peak = fp8_peaks(peaks, src, ms * 1e-3, clk.get("sm_mhz"), num_sms)
    gemm_tf = step_flops() * args.steps / (kernel_ms["gemm"] * 1e-3) / 1e12
    cbytes = cast_bytes(transposed=args.transposed_copies)
    cast_gbs = cbytes * args.steps / (kernel_ms["cast"] * 1e-3) / 1e9
    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8(e4m3,e5m2) x fp8 -> fp32 accumulate, bf16 out",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights, log-uniform signed grads)",
        "config": {
            "workload": WORKLOAD,
            "tokens": TOKENS, "hidden": 4096, "ffn": 16384,
            "layers": [f"{n} {fi}->{fo}" for n, fi, fo in layers()],
            "recipe": "HYBRID delayed scaling, amax_history_len=16, max",
            "gflop_per_step": round(step_flops() / 1e9, 1),
            "cast_bytes_per_step": cbytes,
            "backward_operands": ("transposed copies from the casts, all operands K-major"
                                  if args.transposed_copies else
                                  "forward codes read MN-major (W in dgrad, dY and X in wgrad); no transposed copies"),
            "l2": "inputs larger than L2 (about 4.3 GB touched per step)",
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "gemm_tflops": round(gemm_tf, 1),
        "cast_gbs": round(cast_gbs, 1),
        "roofline": {
            "bound": "tensor",
            "achieved": round(gemm_tf, 1),
            "peak": round(fp8_peak, 1),
            "unit": "TFLOP/s",
            "frac": round(gemm_tf / fp8_peak, 4),
            "traffic": gemm_traffic(),
            "traffic_unit": "bytes per GEMM launch (dram read + write, ncu), mean of the step's 12",
            "algorithmic_bytes": sum(gemm_algorithmic_bytes()) // len(layers()) // 3,
            "peak_source": peak_how + " -- dense FP8 = 2 x dense bf16",
            "nominal_per_clock": None if clock_peak is None else {
                "peak": round(clock_peak, 1), "frac": round(gemm_tf / clock_peak, 4),
                "how": f"{num_sms} SMs x {FP8_FLOP_PER_SM_CLOCK} FP8 FLOP/clock x median SM clock "
                       f"{clk.get('sm_mhz')} MHz of the timed region"},
        },
        "gemm_fc2": fc2,
        "roofline_cast": {
            "bound": "hbm",
            "achieved": round(cast_gbs, 1),
            "peak": peaks["hbm_gbs"],
            "unit": "GB/s",
            "frac": round(cast_gbs / peaks["hbm_gbs"], 4),
            "peak_source": f"hbm_gbs ({src})",
        },
        "kernel_ms_per_step": {k: round(v / args.steps, 4) for k, v in kernel_ms.items()},
        "kernel_windows": f"a second pass of the same {args.steps} steps with a CUDA event pair around each kernel "
                          f"kind: {round(ms_events / args.steps, 4)} ms/step with the events, "
                          f"{round(ms / args.steps, 4)} without",
        "cast_sweep": sweep,
        "mx_step": mx,
        "layer_step": chained,
        "e2e": e2e,
        "gpu_launches": step.launches_per_step() * args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_sample_tokens)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def gemm_fc2(step, s, device_index, peaks, src, num_sms, launches=30, warmup=10):
    """The FC2 forward GEMM alone, M x N x K = 8192 x 4096 x 16384, E4M3 x E4M3
    -> bf16, on the step's cast codes of FC2's X and W: `launches` back-to-back
    launches between two CUDA events on the launching stream, after `warmup`.
    The operands (201 MB of codes) exceed L2, so no flush is needed.  The frac
    uses the burst peak (the region is far shorter than a second)."""
    li = [name for name, _, _ in layers()].index("fc2")
    M, K = step.xq[li].shape
    N = step.wq[li].shape[0]
    for _ in range(warmup):
        step.forward(li, s)
    torch.cuda.synchronize()
    clocks = ClockSampler(device_index)
    clocks.start()
    time.sleep(0.3)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s)
    for _ in range(launches):
        step.forward(li, s)
    b.record(s)
    torch.cuda.synchronize()
    clk = clocks.stop()
    step.R.check_device_error()
    ms = a.elapsed_time(b) / launches
    tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
    peak, how, clock_peak = fp8_peaks(peaks, src, ms * launches * 1e-3, clk.get("sm_mhz"), num_sms)
    return {"shape": f"{M}x{N}x{K}", "operands": "E4M3 x E4M3 -> bf16, the step's FC2 codes (X K-major, W K-major)",
            "launches": launches, "ms_per_launch": round(ms, 4), "tflops": round(tf, 1),
            "peak": round(peak, 1), "frac": round(tf / peak, 4), "peak_source": how,
            "nominal_per_clock": None if clock_peak is None else {
                "peak": round(clock_peak, 1), "frac": round(tf / clock_peak, 4),
                "how": f"{num_sms} SMs x {FP8_FLOP_PER_SM_CLOCK} FP8 FLOP/clock x median SM clock "
                       f"{clk.get('sm_mhz')} MHz sampled around the launches"},
            "clocks": clk,
            "library_reference": library_fc2(step, s, li, launches, warmup)}


def library_fc2(step, s, li, launches, warmup):
    """A library reference beside the FC2 figure (not a denominator, and not on
    the path): torch._scaled_mm -- cuBLASLt's FP8 GEMM -- on the same E4M3
    codes, timed the same way.  Null fields with the reason when this torch
    build or GPU does not offer it."""
    try:
        a = step.xq[li].view(torch.float8_e4m3fn)
        b = step.wq[li].view(torch.float8_e4m3fn)
        one = torch.ones((), dtype=torch.float32, device=a.device)

        def run():
            return torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

        for _ in range(warmup):
            run()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(launches):
            run()
        e1.record(s)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / launches
        M, K = a.shape
        N = b.shape[0]
        return {"what": "torch._scaled_mm (cuBLASLt FP8), same codes, bf16 out", "ms_per_launch": round(ms, 4),
                "tflops": round(2.0 * M * N * K / (ms * 1e-3) / 1e12, 1)}
    except (RuntimeError, AttributeError, TypeError) as e:
        return {"what": "torch._scaled_mm (cuBLASLt FP8)", "unavailable": str(e).splitlines()[0][:200]}


def aggregate(ms, work_per_rank, world, device):
    """Whole-job figure of a replicas run: the slowest rank's time (max over
    ranks) and every rank's work over it.  Returns (ms_max, TFLOP/s)."""
    import torch.distributed as dist

    ms_t = torch.tensor([float(ms)], device=device, dtype=torch.float64)
    if world > 1:
        dist.all_reduce(ms_t, op=dist.ReduceOp.MAX)
    ms_max = float(ms_t.item())
    return ms_max, work_per_rank * world / (ms_max * 1e-3) / 1e12


def cast_sweep(fp8, device, hbm_gbs, reps=5):
    """The standalone amax+cast sweep: bf16 tensors of 2^20, 2^24, 2^28 elements
    (N(0,1) with 0.1% of positions x100), E4M3 and E5M2, delayed scaling (one
    pass, 3 B/element) and current scaling (two passes, 5 B/element).  Each
    launch is timed alone with CUDA events after an L2 flush: a 1 GiB write,
    then a 512 MiB read, so that L2 holds clean lines of an unrelated buffer
    (without the read, the timed launch also pays for writing back the flush's
    dirty lines).  The flush is long enough that the host has enqueued the
    events and the launch before the GPU reaches them, so host launch latency
    stays out of the measurement.  Beside each size, a plain device copy of the
    same bf16 tensor (2 B read + 2 B written per element) is timed the same way:
    the rate one launch of that size reaches.  Every entry gives its fraction of
    the measured HBM copy peak hbm_gbs, and each cast its time against that
    copy's (copy_time_ratio = copy us / cast us: at sizes the L2 holds, both
    kernels are bound by reading the same 2 B per element from DRAM)."""
    from fp8_mixed_precision_history_gb300 import synthetic

    flush = torch.empty(1 << 30, dtype=torch.uint8, device=device)
    clean = torch.ones(1 << 29, dtype=torch.uint8, device=device)
    sink = torch.empty((), dtype=torch.int64, device=device)
    s = torch.cuda.current_stream()

    def timed(fn):
        tot = 0.0
        for _ in range(reps):
            flush.fill_(1)
            torch.sum(clean.view(torch.int64), dim=0, out=sink)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(s)
            fn()
            b.record(s)
            b.synchronize()
            tot += a.elapsed_time(b)
        return tot / reps

    out = {"flush": "1 GiB write, then 512 MiB read", "peak_gbs": hbm_gbs}
    for log2n in (20, 24, 28):
        n = 1 << log2n
        x = synthetic.spiky((n,), 2000 + log2n, device=device)
        q = torch.empty(n, dtype=torch.uint8, device=device)
        y = torch.empty_like(x)
        ms = timed(lambda: y.copy_(x))
        gbs = 4 * n / (ms * 1e-3) / 1e9
        copy_ms = ms
        out[f"2^{log2n}_copy"] = {"us": round(ms * 1e3, 2), "gbs": round(gbs, 1), "frac": round(gbs / hbm_gbs, 4)}
        del y
        for fmt, fname in ((fp8.E4M3, "e4m3"), (fp8.E5M2, "e5m2")):
            R = fp8.Recipe(1)
            R.quantize(0, x, fmt, fp8.CURRENT, out=q, stream=s)  # warm start (history gets an amax)
            R.update_scales(s)
            for mode, mname, bpe in ((fp8.DELAYED, "delayed", 3), (fp8.CURRENT, "current", 5)):
                ms = timed(lambda: R.quantize(0, x, fmt, mode, out=q, stream=s))
                gbs = bpe * n / (ms * 1e-3) / 1e9
                out[f"2^{log2n}_{fname}_{mname}"] = {"us": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                                                    "frac": round(gbs / hbm_gbs, 4),
                                                    "copy_time_ratio": round(copy_ms / ms, 3)}
            R.check_device_error()
            R.close()
        del x, q
    return out


def mx_step(fp8, device, steps=30, warmup=3):
    """The same transformer-layer step with MX block scaling instead of the
    per-tensor recipe: per layer, MX-quantise X and W (E4M3) and dY (E5M2),
    each with its transposed copy, then the forward, dgrad and wgrad MX GEMMs
    (bf16 out).  No scale state is kept: the block scales travel with the
    codes.  Returns the step's TFLOP/s and the kernel split (CUDA events)."""
    from fp8_mixed_precision_history_gb300 import synthetic

    s = torch.cuda.current_stream()
    R = fp8.Recipe(1)
    bufs = []
    for li, (_, fin, fout) in enumerate(layers()):
        x = synthetic.normal((TOKENS, fin), 1.0, 7000 + 10 * li, device=device)
        w = synthetic.normal((fout, fin), 0.02, 7001 + 10 * li, device=device)
        dy = synthetic.grad_like((TOKENS, fout), 7002 + 10 * li, device=device)
        qx = R.mx_quantize(x, fp8.E4M3, transpose=True)
        qw = R.mx_quantize(w, fp8.E4M3, transpose=True)
        qd = R.mx_quantize(dy, fp8.E5M2, transpose=True)
        outs = (torch.empty((TOKENS, fout), dtype=torch.bfloat16, device=device),
                torch.empty((TOKENS, fin), dtype=torch.bfloat16, device=device),
                torch.empty((fout, fin), dtype=torch.bfloat16, device=device))
        bufs.append((x, w, dy, qx, qw, qd, outs))

    def quant(src, dt, q):
        fp8.fp8_mx_quantize(R.handle, src, src.shape[0], src.shape[1], dt, q[0], q[1], q[2], q[3], s)

    ev = {"quant": [], "gemm": []}

    def timed(kind, fn, record):
        if not record:
            fn()
            return
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s)
        fn()
        b.record(s)
        ev[kind].append((a, b))

    def one(record):
        for x, w, dy, qx, qw, qd, (y, dx, dw) in bufs:
            timed("quant", lambda: (quant(x, fp8.E4M3, qx), quant(w, fp8.E4M3, qw)), record)
            timed("gemm", lambda: R.mx_gemm(qx[0], fp8.E4M3, qx[1], qw[0], fp8.E4M3, qw[1], out=y, stream=s),
                  record)
        for x, w, dy, qx, qw, qd, (y, dx, dw) in reversed(bufs):
            timed("quant", lambda: quant(dy, fp8.E5M2, qd), record)
            timed("gemm", lambda: R.mx_gemm(qd[0], fp8.E5M2, qd[1], qw[2], fp8.E4M3, qw[3], out=dx, stream=s),
                  record)
            timed("gemm", lambda: R.mx_gemm(qd[2], fp8.E5M2, qd[3], qx[2], fp8.E4M3, qx[3], out=dw, stream=s),
                  record)

    for _ in range(warmup):
        one(False)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s)
    for _ in range(steps):
        one(False)
    t1.record(s)
    torch.cuda.synchronize()
    for _ in range(steps):  # the split: a second pass with events around each kernel kind
        one(True)
    torch.cuda.synchronize()
    R.check_device_error()
    ms = t0.elapsed_time(t1) / steps
    split = {k: round(sum(a.elapsed_time(b) for a, b in v) / steps, 4) for k, v in ev.items()}
    qbytes = sum((4.0 + 2.0 / 32) * n for _, fin, fout in layers() for n in (TOKENS * fin, fout * fin, TOKENS * fout))
    R.close()
    return {"value": round(step_flops() / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "steps": steps, "kernel_ms_per_step": split,
            "gemm_tflops": round(step_flops() / (split["gemm"] * 1e-3) / 1e12, 1),
            "quant_gbs": round(qbytes / (split["quant"] * 1e-3) / 1e9, 1),
            "what": "MX block scaling (32-element E8M0 scales), same layers, tokens and launch order"}


def run_e2e(step, s, args):
    """Same step through the same C-ABI calls, with every step's inputs (X, W,
    dY of the four layers) copied in from pinned host memory and its outputs
    (Y, dX, dW) copied back, inside the timed region.  The copies are
    pipelined against the kernels: one stream uploads, the compute stream runs
    the step, one stream downloads; per-layer events order them, so layer l+1's
    inputs arrive while layer l computes and finished outputs leave while later
    layers compute.  Device input/output buffers alternate between two sets so
    that step k+1's uploads never overwrite what step k still reads."""
    hx = [t.cpu().pin_memory() for t in step.x]
    hw = [t.cpu().pin_memory() for t in step.w]
    hd = [t.cpu().pin_memory() for t in step.dy]
    hy = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in step.y]
    hdx = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in step.dx]
    hdw = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in step.dw]
    h2d = sum(t.numel() * t.element_size() for t in hx + hw + hd)
    d2h = sum(t.numel() * t.element_size() for t in hy + hdx + hdw)
    names = ("x", "w", "dy", "y", "dx", "dw")
    sets = [{n: list(getattr(step, n)) for n in names},
            {n: [torch.empty_like(t) for t in getattr(step, n)] for n in names}]
    up = torch.cuda.Stream(device=s.device)
    down = torch.cuda.Stream(device=s.device)
    L = len(step.x)
    fp8 = step.fp8
    free_in = [None, None]    # compute finished reading a set's inputs
    free_out = [None, None]   # download finished reading a set's outputs

    def ev(stream):
        e = torch.cuda.Event()
        e.record(stream)
        return e

    def one(k):
        b = k % 2
        cur = sets[b]
        for n in names:
            setattr(step, n, cur[n])
        # uploads of this step's inputs, in the order compute needs them
        if free_in[b] is not None:
            up.wait_event(free_in[b])
        in_fwd, in_bwd = [], [None] * L
        with torch.cuda.stream(up):
            for li in range(L):
                cur["x"][li].copy_(hx[li], non_blocking=True)
                cur["w"][li].copy_(hw[li], non_blocking=True)
                in_fwd.append(ev(up))
            for li in reversed(range(L)):
                cur["dy"][li].copy_(hd[li], non_blocking=True)
                in_bwd[li] = ev(up)
        # compute
        if free_out[b] is not None:
            s.wait_event(free_out[b])
        y_done, bwd_done = [], [None] * L
        for li in range(L):
            s.wait_event(in_fwd[li])
            step._casts(li, fp8.DELAYED, s, ("x", "w"))
            step.forward(li, s)
            y_done.append(ev(s))
        for li in reversed(range(L)):
            s.wait_event(in_bwd[li])
            step._casts(li, fp8.DELAYED, s, ("dy",))
            step.dgrad(li, s)
            step.wgrad(li, s)
            bwd_done[li] = ev(s)
        step.R.update_scales(s)
        free_in[b] = ev(s)
        # downloads of this step's results
        with torch.cuda.stream(down):
            for li in range(L):
                down.wait_event(y_done[li])
                hy[li].copy_(cur["y"][li], non_blocking=True)
            for li in reversed(range(L)):
                down.wait_event(bwd_done[li])
                hdx[li].copy_(cur["dx"][li], non_blocking=True)
                hdw[li].copy_(cur["dw"][li], non_blocking=True)
            free_out[b] = ev(down)

    for k in range(max(2, args.warmup)):
        one(k)
    torch.cuda.synchronize()
    # Three windows of n steps each; the value is the median window.  The host
    # link is shared with whatever else the host runs, so one window can
    # catch another job's transfers; every window is reported.
    n = max(2, min(args.steps, 10))
    windows = []
    k0 = max(2, args.warmup)
    for _ in range(3):
        a = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        a.record(s)
        up.wait_event(a)
        down.wait_event(a)
        for k in range(k0, k0 + n):
            one(k)
        s.wait_event(free_out[(k0 + n - 1) % 2])
        e.record(s)
        torch.cuda.synchronize()
        windows.append(a.elapsed_time(e) / n)
        k0 += n
    for nm in names:  # leave the step on its first buffer set
        setattr(step, nm, sets[0][nm])
    ms = sorted(windows)[1]
    return {"value": round(step_flops() / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3),
            "steps": n, "windows_ms_per_step": [round(w, 3) for w in windows],
            "timing": f"median of 3 windows of {n} steps",
            "overlap": "uploads, kernels and downloads on three streams"}


# --------------------------------------------------------- oracle (CPU) --

_ORACLE_INPUTS = {}


def oracle_inputs(tokens, out_div):
    """X, W, dY of every layer for an oracle sample: `tokens` tokens and each
    layer's output features divided by out_div (at least 16); drawn once per
    size and kept, so that repeated samples time the oracle only."""
    from fp8_mixed_precision_history_gb300 import synthetic

    key = (tokens, out_div)
    if key not in _ORACLE_INPUTS:
        _ORACLE_INPUTS.clear()
        inputs = []
        for li, (_, fin, fout) in enumerate(layers()):
            fo = max(16, fout // out_div)
            x = synthetic.bits(synthetic.normal((tokens, fin), 1.0, 7000 + 10 * li))
            w = synthetic.bits(synthetic.normal((fo, fin), 0.02, 7000 + 10 * li + 1))
            dy = synthetic.bits(synthetic.grad_like((tokens, fo), 7000 + 10 * li + 2))
            inputs.append((x, w, dy))
        _ORACLE_INPUTS[key] = inputs
    return _ORACLE_INPUTS[key]


def oracle_step_sample(tokens, out_div=1):
    """The oracle on the same step with `tokens` tokens and every layer's output
    features divided by out_div (1: all weights full size): casts of X, W, dY,
    then forward, dgrad and wgrad GEMMs of every layer.  Returns (flop done,
    seconds)."""
    import numpy as np

    import oracle

    inputs = oracle_inputs(tokens, out_div)
    R = oracle.DelayedRecipe(4 * len(inputs))
    flop = 0
    t0 = time.perf_counter()
    for li, (x, w, dy) in enumerate(inputs):
        xq = R.quantize(4 * li, x, oracle.E4M3, current=True)
        wq = R.quantize(4 * li + 1, w, oracle.E4M3, current=True)
        dq = R.quantize(4 * li + 2, dy, oracle.E5M2, current=True)
        sx, sw, sd = (np.float32(R.t[4 * li + k].cast_scale_inv) for k in range(3))
        oracle.gemm(xq, oracle.E4M3, wq, oracle.E4M3, sx * sw, want_abs=False)
        oracle.gemm(dq, oracle.E5M2, np.ascontiguousarray(wq.T), oracle.E4M3, sd * sw, want_abs=False)
        oracle.gemm(np.ascontiguousarray(dq.T), oracle.E5M2, np.ascontiguousarray(xq.T), oracle.E4M3,
                    sd * sx, want_abs=False)
        fin, fout = x.shape[1], dy.shape[1]
        flop += 3 * 2 * tokens * fin * fout
    R.update()
    return flop, time.perf_counter() - t0


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def oracle_sample_size(seconds):
    """(tokens, out_div) of an oracle sample that takes about `seconds` on these
    cores.  A step at 8 tokens gives the step's fixed cost (the weight casts,
    the weight-gradient outputs); where that alone exceeds `seconds`, every
    layer's output features are divided by a power of two instead.  Otherwise
    a step at 32 tokens gives the cost per token.  The calibration steps also
    serve as warm-up."""
    _, t8 = oracle_step_sample(8)
    if t8 > seconds:
        div = 1
        while div < 256 and t8 / div > seconds:
            div *= 2
        return 8, div
    _, t32 = oracle_step_sample(32)
    per_token = max((t32 - t8) / 24, 1e-6)
    fixed = max(t8 - 8 * per_token, 0.0)
    return max(8, min(TOKENS, int((seconds - fixed) / per_token) // 8 * 8)), 1


def sample_text(tokens, out_div):
    return f"{tokens} tokens instead of {TOKENS}" + (
        f", every layer's output features / {out_div}" if out_div > 1 else "")


CPU_BASELINE_SECONDS = 12.0   # the oracle sample timed beside the GPU bench
REFERENCE_SECONDS = 120.0     # all timed steps of `--impl reference` together


def cpu_baseline(tokens):
    import oracle

    oracle.set_num_threads(cpu_cores())
    out_div = 1
    if tokens is None:
        tokens, out_div = oracle_sample_size(CPU_BASELINE_SECONDS)
    flop, sec = oracle_step_sample(tokens, out_div)
    return {"value": round(flop / sec / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"the full step (4 layers: casts, fwd, dgrad, wgrad) at {sample_text(tokens, out_div)}; "
                      f"{flop / 1e9:.1f} GFLOP in {sec:.2f} s"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    # every host core: the other ranks do no work (a launcher may have set
    # OMP_NUM_THREADS=1 for each rank)
    oracle.set_num_threads(cpu_cores())
    # each timed step a sample sized so that all of them take about
    # REFERENCE_SECONDS (at most CPU_BASELINE_SECONDS each)
    tokens, out_div = args.cpu_sample_tokens, 1
    if tokens is None:
        tokens, out_div = oracle_sample_size(min(CPU_BASELINE_SECONDS, REFERENCE_SECONDS / max(1, args.steps)))
    for _ in range(args.warmup):
        oracle_step_sample(tokens, out_div)
    times, flop = [], 0
    for _ in range(args.steps):
        flop, sec = oracle_step_sample(tokens, out_div)
        times.append(sec)
    total = sum(times)
    value = flop * len(times) / total / 1e12
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1000 * total / len(times), 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens": TOKENS, "sample_tokens": tokens, "sample_out_div": out_div},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"full step at {sample_text(tokens, out_div)} per timed step "
                                   f"({flop / 1e9:.1f} GFLOP); {total:.1f} s in all"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


LOOP_TOKENS = 16384
LOOP_STEPS = 32
LOOP_SPIKE = 20


def run_loop(args):
    """The 32-step delayed-scaling training loop at 16384 tokens: the four layers
    of the step, HYBRID recipe with a 16-entry "max" history, activations
    drifting x1.05 per step with a x50 spike at step 20, fixed weights, fresh
    gradients every step.  Each step is timed with CUDA events around its
    launches (casts, forward, dgrad, wgrad, scale update; input generation stays
    outside).  After every step each tensor's state is appended to the JSONL file
    args.loop32: amax, next scale, and the step's saturated and underflowed
    counts.  Prints one JSON summary line."""
    import fp8_mixed_precision_history_gb300 as fp8
    from fp8_mixed_precision_history_gb300 import synthetic

    fp8.load()
    dev = torch.device("cuda", 0)
    T = LOOP_TOKENS
    L = layers()
    R = fp8.Recipe(4 * len(L), amax_history_len=16)
    s = torch.cuda.current_stream()

    def x_of(step, li, fin):
        std = 1.05 ** step * (50.0 if step == LOOP_SPIKE else 1.0)
        return synthetic.normal((T, fin), std, synthetic.seed_for(5, li, "x", step), device=dev)

    def dy_of(step, li, fout):
        return synthetic.grad_like((T, fout), synthetic.seed_for(5, li, "dy", step), device=dev)

    W = [synthetic.normal((fout, fin), 0.02, synthetic.seed_for(5, li, "w"), device=dev)
         for li, (_, fin, fout) in enumerate(L)]
    u8 = dict(dtype=torch.uint8, device=dev)
    bf = dict(dtype=torch.bfloat16, device=dev)
    xq = [torch.empty((T, fin), **u8) for _, fin, _ in L]
    wq = [torch.empty((fout, fin), **u8) for _, fin, fout in L]
    dq = [torch.empty((T, fout), **u8) for _, _, fout in L]
    y = [torch.empty((T, fout), **bf) for _, _, fout in L]
    dx = [torch.empty((T, fin), **bf) for _, fin, _ in L]
    dw = [torch.empty((fout, fin), **bf) for _, fin, fout in L]
    # warm start: a current-scaling pass over step 0's tensors, then an update
    for li, (_, fin, fout) in enumerate(L):
        R.quantize(4 * li, x_of(0, li, fin), fp8.E4M3, fp8.CURRENT, out=xq[li], stream=s)
        R.quantize(4 * li + 1, W[li], fp8.E4M3, fp8.CURRENT, out=wq[li], stream=s)
        R.quantize(4 * li + 2, dy_of(0, li, fout), fp8.E5M2, fp8.CURRENT, out=dq[li], stream=s)
    R.update_scales(s)
    torch.cuda.synchronize()
    flop = 3 * 2.0 * T * sum(fin * fout for _, fin, fout in L)
    names = ("x", "w", "dy", "y")
    step_ms, records = [], []
    for step in range(LOOP_STEPS):
        xs = [x_of(step, li, fin) for li, (_, fin, _) in enumerate(L)]
        dys = [dy_of(step, li, fout) for li, (_, _, fout) in enumerate(L)]
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s)
        for li in range(len(L)):
            R.quantize(4 * li, xs[li], fp8.E4M3, fp8.DELAYED, out=xq[li], stream=s)
            R.quantize(4 * li + 1, W[li], fp8.E4M3, fp8.DELAYED, out=wq[li], stream=s)
            R.gemm(4 * li, xq[li], fp8.E4M3, 4 * li + 1, wq[li], fp8.E4M3, out=y[li], amax_out_id=4 * li + 3,
                   stream=s)
        for li in reversed(range(len(L))):
            R.quantize(4 * li + 2, dys[li], fp8.E5M2, fp8.DELAYED, out=dq[li], stream=s)
            R.gemm(4 * li + 2, dq[li], fp8.E5M2, 4 * li + 1, wq[li], fp8.E4M3, out=dx[li], stream=s,
                   b_major=fp8.MN_MAJOR)
            R.gemm(4 * li + 2, dq[li], fp8.E5M2, 4 * li, xq[li], fp8.E4M3, out=dw[li], stream=s,
                   a_major=fp8.MN_MAJOR, b_major=fp8.MN_MAJOR)
        R.update_scales(s)
        b.record(s)
        torch.cuda.synchronize()
        R.check_device_error()
        step_ms.append(a.elapsed_time(b))
        for li, (name, _, _) in enumerate(L):
            for k, kind in enumerate(names):
                st, _ = R.get_state(4 * li + k)
                records.append({"step": step, "layer": name, "tensor": kind, "amax": st["amax_last"],
                                "scale": st["scale"], "scale_inv": st["scale_inv"],
                                "n_saturated": st["n_saturated_last"], "n_underflow": st["n_underflow_last"]})
        del xs, dys
    R.close()
    with open(args.loop32, "w") as f:
        for r in records:
            f.write(json.dumps(r) + "\n")
    per_step = lambda kind, key: [sum(r[key] for r in records if r["step"] == t and r["tensor"] == kind)
                                  for t in range(LOOP_STEPS)]
    med = statistics.median(step_ms)
    print(json.dumps({
        "case": "loop32", "tokens": T, "steps": LOOP_STEPS, "spike_step": LOOP_SPIKE,
        "ms_per_step": {"median": round(med, 4), "min": round(min(step_ms), 4), "max": round(max(step_ms), 4)},
        "tflops_median": round(flop / (med * 1e-3) / 1e12, 1),
        "x_saturated_per_step": per_step("x", "n_saturated"),
        "x_underflow_per_step": per_step("x", "n_underflow"),
        "states": args.loop32, "records": len(records)}), flush=True)


def run_case(args):
    """One kernel on a profiling-sized case (inputs larger than L2, a few
    hundred MB on the device):
      gemm    one of the step's GEMMs (--gemm, default fc2_fwd: M=8192, N=4096,
              K=16384, E4M3 x E4M3 -> bf16) in the step's operand layouts
      cast    flat delayed cast of 2^26 (--cast-log2n) bf16 elements to E4M3
      cast_t  delayed cast + transpose of X [8192, 16384] to E4M3
      mx_gemm MX block-scaled GEMM, same shape, E4M3 x E4M3 -> bf16
      mx_quant MX quantisation of X [8192, 16384] to E4M3 with its transposed
              copy (4 B/element + 2 x 1/32 B of block scales)
      grad_ar one rank's device work in an 8-rank FP8 gradient all-reduce of the
              FC1 weight gradient (16384 x 4096): amax, E5M2 quantise, exact
              reduce of 8 chunks, dequantise -- 2 + 3 + (1 + 1/8) + 3 B/element
    Prints the CUDA-event time per launch."""
    import fp8_mixed_precision_history_gb300 as fp8
    from fp8_mixed_precision_history_gb300 import synthetic

    fp8.load()
    dev = torch.device("cuda", 0)
    R = fp8.Recipe(3)
    s = torch.cuda.current_stream()
    if args.case == "gemm":
        layer, kind = args.gemm.split("_")
        _, fin, fout = [l for l in layers() if l[0] == layer][0]
        T = TOKENS
        xq = R.quantize(0, synthetic.normal((T, fin), 1.0, 11, device=dev), fp8.E4M3, fp8.CURRENT)
        wq = R.quantize(1, synthetic.normal((fout, fin), 0.02, 12, device=dev), fp8.E4M3, fp8.CURRENT)
        dq = R.quantize(2, synthetic.grad_like((T, fout), 13, device=dev), fp8.E5M2, fp8.CURRENT)
        # (a_id, A, a_dtype, a_major, b_id, B, b_dtype, b_major, M, N, K): the step's layouts
        g = {"fwd": (0, xq, fp8.E4M3, fp8.K_MAJOR, 1, wq, fp8.E4M3, fp8.K_MAJOR, T, fout, fin),
             "dgrad": (2, dq, fp8.E5M2, fp8.K_MAJOR, 1, wq, fp8.E4M3, fp8.MN_MAJOR, T, fin, fout),
             "wgrad": (2, dq, fp8.E5M2, fp8.MN_MAJOR, 0, xq, fp8.E4M3, fp8.MN_MAJOR, fout, fin, T)}[kind]
        M, N, K = g[8], g[9], g[10]
        odt = {"bf16": fp8.OUT_BF16, "e4m3": fp8.OUT_E4M3, "e5m2": fp8.OUT_E5M2}[args.gemm_out]
        out = torch.empty((M, N), dtype=torch.bfloat16 if odt == fp8.OUT_BF16 else torch.uint8, device=dev)
        act = {"none": fp8.ACT_NONE, "gelu": fp8.ACT_GELU, "dgelu": fp8.ACT_DGELU}[args.gemm_act]
        aux = None
        if act == fp8.ACT_DGELU or (act == fp8.ACT_GELU and not args.gemm_no_aux):
            # values like FC1's output (GELU writes its derivative there)
            aux = synthetic.normal((M, N), 1.2, 14, device=dev)
        if odt != fp8.OUT_BF16:
            R.set_state(2, [1.0] * 16, 64.0, odt - 2)
        work = 2.0 * M * N * K
        unit = "TFLOP/s"

        def launch():
            R.gemm(g[0], g[1], g[2], g[4], g[5], g[6], out=out, out_dtype=odt, stream=s, a_major=g[3],
                   b_major=g[7], act=act, aux=aux, amax_out_id=2 if odt != fp8.OUT_BF16 else -1)
    elif args.case == "mx_gemm":
        M, N, K = 8192, 4096, 16384
        xq, xs = R.mx_quantize(synthetic.normal((M, K), 1.0, 11, device=dev), fp8.E4M3)
        wq, ws = R.mx_quantize(synthetic.normal((N, K), 0.02, 12, device=dev), fp8.E4M3)
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        work = 2.0 * M * N * K
        unit = "TFLOP/s"

        def launch():
            R.mx_gemm(xq, fp8.E4M3, xs, wq, fp8.E4M3, ws, out=out, stream=s)
    elif args.case == "mx_quant":
        x = synthetic.normal((8192, 16384), 1.0, 14, device=dev)
        unit = "GB/s"
        work = (4.0 + 2.0 / 32) * x.numel()
        bufs = R.mx_quantize(x, fp8.E4M3, transpose=True)

        def launch():
            fp8.fp8_mx_quantize(R.handle, x, x.shape[0], x.shape[1], fp8.E4M3, bufs[0], bufs[1], bufs[2],
                                bufs[3], s)
    elif args.case == "grad_ar":
        from fp8_mixed_precision_history_gb300.grad_allreduce import chunk_size

        world, n = 8, 16384 * 4096
        chunk = chunk_size(n, world)
        g = synthetic.grad_like((n,), 15, device=dev)
        amax = torch.empty(1, dtype=torch.float32, device=dev)
        codes = torch.empty(world * chunk, dtype=torch.uint8, device=dev)
        scale = torch.empty(2, dtype=torch.float32, device=dev)
        red = torch.empty(chunk, dtype=torch.uint8, device=dev)
        out = torch.empty(n, dtype=torch.bfloat16, device=dev)
        unit = "GB/s"
        work = 2.0 * n + 2.0 * n + world * chunk + world * chunk + chunk + n + 2.0 * n

        def launch():
            fp8.fp8_grad_amax(g, n, amax, s)
            fp8.fp8_grad_quantize(g, n, amax, world, codes, world * chunk, scale, s)
            fp8.fp8_grad_reduce(codes, world, chunk, red, s)  # the received [world][chunk] codes
            fp8.fp8_grad_dequantize(codes, n, scale, world, 0, out, s)  # the gathered codes
    else:
        if args.case == "cast":
            if args.cast_draw == "spiky":  # the sweep's tensors: N(0,1) with 0.1 % of positions x100
                x = synthetic.spiky((1 << args.cast_log2n,), 2000 + args.cast_log2n, device=dev)
            else:
                x = synthetic.normal((1 << args.cast_log2n,), 1.0, 13, device=dev)
            q = torch.empty(x.shape, dtype=torch.uint8, device=dev)
            qt = None
            work = 3.0 * x.numel()
        else:
            x = synthetic.normal((8192, 16384), 1.0, 14, device=dev)
            q = torch.empty(x.shape, dtype=torch.uint8, device=dev)
            qt = torch.empty((16384, 8192), dtype=torch.uint8, device=dev)
            work = 4.0 * x.numel()
        unit = "GB/s"
        cfmt = fp8.E5M2 if args.cast_fmt == "e5m2" else fp8.E4M3
        R.quantize(0, x, cfmt, fp8.CURRENT)
        mode = fp8.CURRENT if args.cast_mode == "current" else fp8.DELAYED
        if mode == fp8.CURRENT:
            work += 2.0 * x.numel()  # the amax pass reads the tensor once more

        def launch():
            R.quantize(0, x, cfmt, mode, out=q, out_t=qt, transpose=qt is not None, stream=s)
    for _ in range(max(1, args.warmup)):
        launch()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    reps = max(1, args.steps)
    a.record(s)
    for _ in range(reps):
        launch()
    b.record(s)
    torch.cuda.synchronize()
    R.check_device_error()
    ms = a.elapsed_time(b) / reps
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    print(json.dumps({"case": args.case if args.case != "gemm" else f"gemm {args.gemm}", "ms_per_launch": round(ms, 4),
                      "achieved": round(work / (ms * 1e-3) / scale, 1), "unit": unit}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-sample-tokens", type=int, default=None,
                    help="tokens of the oracle's step sample (default: sized to about 12 s of CPU work, "
                         "and for --impl reference to about 120 s over all timed steps)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-mx", action="store_true", help="skip the MX block-scaling step")
    ap.add_argument("--no-chain", action="store_true", help="skip the chained transformer-layer step")
    ap.add_argument("--transposed-copies", action="store_true",
                    help="casts also write transposed codes and every GEMM operand is K-major")
    ap.add_argument("--case", choices=["gemm", "cast", "cast_t", "mx_gemm", "mx_quant", "grad_ar"],
                    help="run one kernel on a small profiling case instead of the step")
    ap.add_argument("--cast-log2n", type=int, default=26, help="elements (log2) of --case cast")
    ap.add_argument("--cast-fmt", default="e4m3", choices=["e4m3", "e5m2"], help="format of --case cast/cast_t")
    ap.add_argument("--cast-draw", default="normal", choices=["normal", "spiky"],
                    help="--case cast input: N(0,1), or the sweep's N(0,1) with 0.1%% of positions x100")
    ap.add_argument("--cast-mode", default="delayed", choices=["delayed", "current"],
                    help="scaling mode of --case cast / cast_t")
    ap.add_argument("--gemm", default="fc2_fwd",
                    help="GEMM of --case gemm: {qkv,proj,fc1,fc2}_{fwd,dgrad,wgrad}")
    ap.add_argument("--gemm-out", default="bf16", choices=["bf16", "e4m3", "e5m2"],
                    help="output of --case gemm (FP8 outputs use a tensor scale of 64)")
    ap.add_argument("--gemm-no-aux", action="store_true",
                    help="--case gemm --gemm-act gelu: do not write the derivative")
    ap.add_argument("--gemm-act", default="none", choices=["none", "gelu", "dgelu"],
                    help="epilogue activation of --case gemm (with a bf16 aux tensor)")
    ap.add_argument("--loop32", metavar="JSONL",
                    help="run the 32-step delayed-scaling loop at 16384 tokens instead; per-step tensor "
                         "states go to this file")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != world:
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch N > 1 GPUs with "
                 f"python -m torch.distributed.run --nproc-per-node {args.gpus} bench.py --gpus {args.gpus}")
    if args.loop32:
        run_loop(args)
    elif args.case:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
