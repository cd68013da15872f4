"""Delayed-scaling recipe bookkeeping of the oracle (test infrastructure only).

Follows [TE] "4.2 Hopper I -- Transformer Engine / FP8":

* S4.2.4 "delayed scaling": the amax of the tensor being cast is not known before
  the cast, so the scale comes from a history of past amaxes (e.g. the max of the
  last N steps) and the tensor is cast in one pass; a spike is seen one step late.
* S4.2.6 recipe: ``amax_history_len=16``, ``amax_compute_algo="max"``,
  HYBRID = E4M3 forward, E5M2 backward; "TE updates the amax internally to set
  the next step's scales".

Readings (pages silent): a step's amax enters the history after the step's own
cast; the history is a window of the last H recorded amaxes (zeros at start);
only tensors that recorded an amax since the last update are rolled; a tensor
cast several times in one step records the max of those amaxes; the
"most_recent" rule (a TE-style option) uses the newest entry instead of the max.
"""
import math

import numpy as np

from . import E4M3, E5M2, amax as _amax, cast as _cast, reciprocal, scale_from_amax

ALGO_MAX = 0
ALGO_MOST_RECENT = 1

FORMAT_HYBRID = 0
FORMAT_E4M3 = 1


def _nan_max(a, b):
    """max that lets NaN win (the reading used for a NaN amax)."""
    a = np.float32(a)
    b = np.float32(b)
    if math.isnan(a) or math.isnan(b):
        return np.float32("nan")
    return a if a >= b else b


class TensorState:
    def __init__(self, history_len):
        self.history = [np.float32(0.0)] * history_len  # oldest first
        self.scale = np.float32(1.0)
        self.scale_inv = np.float32(1.0)
        self.cast_scale = np.float32(1.0)
        self.cast_scale_inv = np.float32(1.0)
        self.amax_pending = np.float32(0.0)
        self.recorded = False
        self.n_saturated = 0
        self.n_underflow = 0
        self.amax_last = np.float32(0.0)
        self.n_saturated_last = 0
        self.n_underflow_last = 0
        self.fmt = E4M3


class DelayedRecipe:
    def __init__(self, num_tensors, history_len=16, algo=ALGO_MAX, recipe_format=FORMAT_HYBRID):
        assert history_len >= 1
        self.H = history_len
        self.algo = algo
        self.recipe_format = recipe_format
        self.t = [TensorState(history_len) for _ in range(num_tensors)]

    # -- state ------------------------------------------------------------
    def set_state(self, tid, history, scale, fmt=E4M3):
        st = self.t[tid]
        h = [np.float32(v) for v in history]
        assert len(h) == self.H
        st.history = h
        st.scale = np.float32(scale)
        st.scale_inv = reciprocal(st.scale)
        st.cast_scale = st.scale
        st.cast_scale_inv = st.scale_inv
        st.amax_pending = np.float32(0.0)
        st.recorded = False
        st.n_saturated = st.n_underflow = 0
        st.fmt = fmt

    def _reduce_history(self, h):
        if self.algo == ALGO_MOST_RECENT:
            return h[-1]
        m = np.float32(0.0)
        for v in h:
            m = _nan_max(m, v)
        return m

    # -- one cast ([TE] S4.2.4) -------------------------------------------
    def quantize(self, tid, x_bits, fmt, current=False, update_now=False):
        """Cast x (bf16 bits) of tensor ``tid``; returns the FP8 codes."""
        if self.recipe_format == FORMAT_E4M3 and fmt != E4M3:
            raise ValueError("E4M3-only recipe casts every tensor to E4M3")
        st = self.t[tid]
        a = _amax(x_bits)
        if current:
            s = scale_from_amax(a, fmt, st.scale)
            sinv = reciprocal(s)
        else:
            s, sinv = st.scale, st.scale_inv
        q, ns, nu = _cast(x_bits, s, fmt)
        st.cast_scale, st.cast_scale_inv = np.float32(s), np.float32(sinv)
        st.amax_pending = _nan_max(st.amax_pending, a)
        st.recorded = True
        st.n_saturated += ns
        st.n_underflow += nu
        st.fmt = fmt
        if update_now:
            self._update_one(tid)
        return q

    def record_cast(self, tid, a, n_saturated, n_underflow, fmt):
        """A cast made outside quantize() with this tensor's delayed scale --
        the next stage's cast composed into a GEMM epilogue ([TE] S4.2.4):
        records its amax (max|value|), counts and cast scale."""
        st = self.t[tid]
        st.cast_scale, st.cast_scale_inv = st.scale, st.scale_inv
        st.amax_pending = _nan_max(st.amax_pending, a)
        st.recorded = True
        st.n_saturated += n_saturated
        st.n_underflow += n_underflow
        st.fmt = fmt

    def record_amax(self, tid, a):
        """An amax measured elsewhere (e.g. of a GEMM output) joins this step's."""
        st = self.t[tid]
        st.amax_pending = _nan_max(st.amax_pending, a)
        st.recorded = True

    # -- end of step ([TE] S4.2.6: next step's scales) -----------------------
    def _update_one(self, tid):
        st = self.t[tid]
        st.history = st.history[1:] + [np.float32(st.amax_pending)]
        m = self._reduce_history(st.history)
        st.scale = scale_from_amax(m, st.fmt, st.scale)
        st.scale_inv = reciprocal(st.scale)
        st.amax_last = st.amax_pending
        st.n_saturated_last, st.n_underflow_last = st.n_saturated, st.n_underflow
        st.amax_pending = np.float32(0.0)
        st.recorded = False
        st.n_saturated = st.n_underflow = 0

    def update(self):
        for tid, st in enumerate(self.t):
            if st.recorded:
                self._update_one(tid)
