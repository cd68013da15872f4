"""Shared helpers of the GPU parity tests (comparison logic only)."""
import numpy as np
import torch

import oracle
from fp8_mixed_precision_history_gb300 import synthetic


def f32_bits(v):
    return int(np.array([v], np.float32).view(np.uint32)[0])


def bf16_ord(bits):
    """bf16 bit patterns -> integers ordered like the values (+0 == -0)."""
    b = np.asarray(bits).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def prefill_for(x_bits, fmt):
    """History of 16 copies of amax(x) and the scale it gives (oracle)."""
    a = float(oracle.amax(x_bits))
    return [a] * 16, float(oracle.scale_from_amax(a, fmt))


def check_state(R, OR, tid, what=""):
    """GPU recipe state of tensor tid == oracle recipe state, bit for bit."""
    st, hist = R.get_state(tid)
    o = OR.t[tid]
    pairs = [("scale", o.scale), ("scale_inv", o.scale_inv), ("cast_scale", o.cast_scale),
             ("cast_scale_inv", o.cast_scale_inv), ("amax_pending", o.amax_pending),
             ("amax_last", o.amax_last)]
    for k, v in pairs:
        assert f32_bits(st[k]) == f32_bits(v), f"{what} {k}: gpu {st[k]!r} oracle {float(v)!r}"
    assert st["n_saturated"] == o.n_saturated, f"{what} n_saturated {st['n_saturated']} vs {o.n_saturated}"
    assert st["n_underflow"] == o.n_underflow, f"{what} n_underflow {st['n_underflow']} vs {o.n_underflow}"
    assert st["n_saturated_last"] == o.n_saturated_last, what
    assert st["n_underflow_last"] == o.n_underflow_last, what
    assert bool(st["recorded"]) == bool(o.recorded), what
    assert [f32_bits(h) for h in hist] == [f32_bits(h) for h in o.history], f"{what} history"


def fp32_mma_rel(K):
    """Error bound of the GEMM's FP32 accumulation, as a fraction of
    sum_k |a*b| * factor, for operands of any distribution.  Each K = 32 MMA
    step rounds twice -- the sum of its 32 exact products to fp32, then that
    sum's add into the TMEM partial -- and either rounding may be directed
    (up to one fp32 ulp, 2^-23 of a magnitude <= the partial's sum|ab|).  A
    partial spans at most 64 steps (K = 2048) before it is added into the
    round-to-nearest fp32 total (2^-24 per add); the output's x factor rounds
    once more (2^-24).  So |D - exact| <= (2 * min(64, ceil(K/32)) * 2^-23
    + (ceil(K/2048) + 1) * 2^-24) * sum|ab| * factor; without the promotion
    every 2048 of K the first term would grow with K."""
    return 2 * min(64, -(-K // 32)) * 2.0 ** -23 + (-(-K // 2048) + 1) * 2.0 ** -24


def check_gemm_sample(D32, Db, A, afmt, B, bfmt, factor, rows, cols=None, rel=1e-6):
    """Compare sampled rows (and columns) of a GPU GEMM output with the oracle.

    D32 / Db: the GPU outputs (torch CUDA tensors, fp32 / bf16) or None.
    A [M, K], B [N, K]: host FP8 codes.  rel: error bound as a fraction of
    sum_k |a*b| * factor.  Returns the worst bf16 ulp distance seen."""
    ri = torch.as_tensor(np.asarray(rows, np.int64), device=D32.device if D32 is not None else Db.device)
    g32 = D32.index_select(0, ri).cpu().numpy() if D32 is not None else None
    gb = to_host_u16(Db.index_select(0, ri)) if Db is not None else None
    acc, absacc, ob = oracle.gemm(A, afmt, B, bfmt, factor, rows=rows)
    worst = _cmp(g32, gb, acc, absacc, ob, factor, rel)
    if cols is not None:
        ci = torch.as_tensor(np.asarray(cols, np.int64), device=ri.device)
        g32 = D32.index_select(1, ci).t().cpu().numpy() if D32 is not None else None
        gb = to_host_u16(Db.index_select(1, ci).t()) if Db is not None else None
        acc, absacc, ob = oracle.gemm(B, bfmt, A, afmt, factor, rows=cols)
        worst = max(worst, _cmp(g32, gb, acc, absacc, ob, factor, rel))
    return worst


def bf16_spacing(v):
    """Distance between adjacent bf16 values around |v| (8-bit significand)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def _cmp(g32, gb, acc, absacc, ob, factor, rel):
    """fp32 output: |gpu - acc*factor| <= rel * sum|ab| * factor.
    bf16 output: the bf16 rounding of a value inside that bound, i.e.
    |gpu - acc*factor| <= bound + one bf16 spacing; where the bound is below half
    a spacing this is 'within 1 ulp of the oracle's bf16', checked as such.
    Both outputs: bf16 == round-to-nearest-even(fp32) bit for bit."""
    f = float(np.float32(factor))
    ref = acc * f
    bound = rel * absacc * f
    worst = 0
    if g32 is not None:
        err = np.abs(g32.astype(np.float64) - ref)
        bad = err > bound
        assert not bad.any(), (f"{int(bad.sum())} fp32 outputs outside {rel:g}*sum|ab|; worst "
                               f"err/bound {float(np.max(err / np.maximum(bound, 1e-300))):.3g}")
    if gb is not None:
        gv = (gb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        sp = bf16_spacing(np.maximum(np.abs(ref), np.abs(gv)))
        bad = np.abs(gv - ref) > bound + sp
        assert not bad.any(), f"{int(bad.sum())} bf16 outputs beyond bound + 1 spacing"
        d = np.abs(bf16_ord(gb) - bf16_ord(ob))
        tight = bound <= 0.5 * bf16_spacing(ref)
        worst = int(d[tight].max()) if tight.any() else 0
        assert worst <= 1, f"bf16 outputs up to {worst} ulp from the oracle where the bound is tight"
    if g32 is not None and gb is not None:
        rn = torch.from_numpy(np.ascontiguousarray(g32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(rn, gb), "bf16 output differs from RN(fp32 output) of the same kernel"
    return worst


def to_host_u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_host_u8(t):
    return synthetic.codes(t)


# ---- MX block scales: the atom layout the C header documents ----------------
def mx_atom_offsets(rows, cols):
    """Byte offset of scale (r, b) for every row r < rows and block b <
    ceil(cols/32):  ((r/128) * ceil(cols/128) + b/4) * 512 + (r%32) * 16
    + ((r/32)%4) * 4 + b%4."""
    nb = (cols + 31) // 32
    ac = (cols + 127) // 128
    r = np.arange(rows, dtype=np.int64)[:, None]
    b = np.arange(nb, dtype=np.int64)[None, :]
    return ((r // 128) * ac + b // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + b % 4


def mx_atoms_from_plain(sc, rows, cols):
    """Plain [rows, ceil(cols/32)] scale codes -> the atom array (padding 0)."""
    size = ((rows + 127) // 128) * ((cols + 127) // 128) * 512
    out = np.zeros(size, np.uint8)
    out[mx_atom_offsets(rows, cols)] = sc
    return out


def mx_plain_from_atoms(atoms, rows, cols):
    """Atom array -> plain [rows, ceil(cols/32)] codes; also checks that every
    padding byte is 0."""
    a = np.asarray(atoms, np.uint8)
    off = mx_atom_offsets(rows, cols)
    pad = np.ones(a.size, bool)
    pad[off.ravel()] = False
    assert not a[pad].any(), "non-zero padding in the scale atoms"
    return a[off]


def check_mx_gemm_sample(D32, Db, A, afmt, sa, B, bfmt, sb, rows, cols=None, rel=1e-6):
    """check_gemm_sample for MX operands (plain scales sa, sb; factor 1)."""
    dev = D32.device if D32 is not None else Db.device
    ri = torch.as_tensor(np.asarray(rows, np.int64), device=dev)
    g32 = D32.index_select(0, ri).cpu().numpy() if D32 is not None else None
    gb = to_host_u16(Db.index_select(0, ri)) if Db is not None else None
    acc, absacc, ob = oracle.mx_gemm(A, afmt, sa, B, bfmt, sb, rows=rows)
    worst = _cmp(g32, gb, acc, absacc, ob, 1.0, rel)
    if cols is not None:
        ci = torch.as_tensor(np.asarray(cols, np.int64), device=dev)
        g32 = D32.index_select(1, ci).t().cpu().numpy() if D32 is not None else None
        gb = to_host_u16(Db.index_select(1, ci).t()) if Db is not None else None
        acc, absacc, ob = oracle.mx_gemm(B, bfmt, sb, A, afmt, sa, rows=cols)
        worst = max(worst, _cmp(g32, gb, acc, absacc, ob, 1.0, rel))
    return worst
