"""FP8 (E5M2) gradient all-reduce on the GPU against the oracle ("FP8 and
low-precision formats", use cases: E5M2 gradient communication; FP8-LM forum
thread: automatic scaling during the all-reduce).

The ranks are emulated in one process on one GPU (grad_allreduce.
all_reduce_local: each rank's kernels run in turn, the exchanges are device
copies).  Every result is compared with the oracle bit for bit: the shared
amax and scale, each rank's codes, the reduced codes and the bf16 output."""
import numpy as np
import pytest
import torch

import oracle
from fp8_mixed_precision_history_gb300 import synthetic
from gpu_util import f32_bits, to_host_u16, to_host_u8

pytestmark = pytest.mark.gpu

E5M2 = oracle.E5M2


def _grads(world, n, seed):
    # gradients of different magnitude per rank, some exact zeros and tiny values
    out = []
    for r in range(world):
        g = synthetic.grad_like((n,), seed + 31 * r, lo=1e-7 * (r + 1), hi=1e-1 * (r + 1))
        out.append(g)
    return out


@pytest.mark.parametrize("world,n,average", [(1, 1000, False), (2, 1, False), (2, 1000, True),
                                             (3, 196615, False), (8, 65536 * 3 + 7, True),
                                             (8, (1 << 22) + 3, False)])
def test_local_all_reduce_matches_oracle(gpu_lib, world, n, average):
    from fp8_mixed_precision_history_gb300 import grad_allreduce

    grads = _grads(world, n, 100 + world + n % 97)
    out, codes = grad_allreduce.all_reduce_local([g.cuda() for g in grads], average=average, with_codes=True)
    torch.cuda.synchronize()
    want, wcodes, _ = oracle.allreduce_e5m2(np.stack([synthetic.bits(g) for g in grads]), average=average)
    got_codes = to_host_u8(codes)
    bad = got_codes != wcodes
    assert not bad.any(), f"{int(bad.sum())} reduced codes differ; first at {np.argwhere(bad)[0]}"
    bad = to_host_u16(out) != want
    assert not bad.any(), f"{int(bad.sum())} outputs differ"


def test_full_size_fc1_weight_gradient(gpu_lib):
    """dW of FC1 (16384 x 4096 = 67M elements) over two ranks."""
    from fp8_mixed_precision_history_gb300 import grad_allreduce

    n = 16384 * 4096
    grads = [synthetic.grad_like((n,), 900 + r) for r in range(2)]
    out, codes = grad_allreduce.all_reduce_local([g.cuda() for g in grads], with_codes=True)
    torch.cuda.synchronize()
    want, wcodes, _ = oracle.allreduce_e5m2(np.stack([synthetic.bits(g) for g in grads]))
    assert np.array_equal(to_host_u8(codes), wcodes)
    assert np.array_equal(to_host_u16(out), want)


@pytest.mark.parametrize("n,padded", [(1037, 3 * 352), (1037, 1043), (5, 13), (8, 8), (70001, 70016)])
def test_steps_one_by_one(gpu_lib, n, padded):
    """amax, the scale, each rank's codes and the zero padding (padded to any
    length, written exactly up to it: the 16 guard bytes after it keep their
    value)."""
    fp8 = gpu_lib
    world = 3
    grads = _grads(world, n, 7 + n)
    a = torch.empty(1, dtype=torch.float32, device="cuda")
    amaxes = []
    for g in grads:
        fp8.fp8_grad_amax(g.cuda(), n, a)
        amaxes.append(float(a.item()))
        assert f32_bits(amaxes[-1]) == f32_bits(oracle.amax(synthetic.bits(g)))
    shared = torch.tensor([max(amaxes)], dtype=torch.float32, device="cuda")
    s_ref = oracle.allreduce_scale(max(amaxes), world)
    for g in grads:
        codes = torch.full((padded + 16,), 0xAB, dtype=torch.uint8, device="cuda")
        scale = torch.empty(2, dtype=torch.float32, device="cuda")
        fp8.fp8_grad_quantize(g.cuda(), n, shared, world, codes, padded, scale)
        torch.cuda.synchronize()
        sc = scale.cpu().numpy()
        assert f32_bits(sc[0]) == f32_bits(s_ref) and f32_bits(sc[1]) == f32_bits(oracle.reciprocal(s_ref))
        q, _, _ = oracle.cast(synthetic.bits(g), s_ref, E5M2)
        c = to_host_u8(codes)
        assert np.array_equal(c[:n], q) and not c[n:padded].any()
        assert (c[padded:] == 0xAB).all(), "a code was written past padded_n"


def _reduce_expected(recv):
    """Exact sum of the decoded codes (float64, -0 kept) encoded once."""
    dec = oracle.decode(recv, E5M2)
    total = dec[0].copy()
    for r in range(1, recv.shape[0]):
        total = total + dec[r]
    return np.array([oracle.encode_double(v, E5M2) for v in total], dtype=np.uint8)


def test_reduce_kernel_edge_cases(gpu_lib):
    """Ties in both directions, sums past 57344, subnormal sums, negative
    zeros, exact cancellations -- and every pair of finite codes."""
    fp8 = gpu_lib
    finite = np.array([c for c in range(256) if (c & 0x7C) != 0x7C], dtype=np.uint8)
    a, b = np.meshgrid(finite, finite, indexing="ij")
    pairs = np.stack([a.ravel(), b.ravel()])  # every pair of finite codes, world = 2
    special = np.array([[0x80, 0x80, 0x7B, 0xFB, 0x01, 0x43, 0x44, 0x3C],
                        [0x80, 0x00, 0x7B, 0xFB, 0x01, 0x43, 0xC4, 0x3D]], np.uint8)
    used = pairs.shape[1] + special.shape[1]
    chunk = -(-used // 16) * 16
    recv = np.zeros((2, chunk), np.uint8)
    recv[:, :pairs.shape[1]] = pairs
    recv[:, pairs.shape[1]:used] = special
    out = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    fp8.fp8_grad_reduce(torch.from_numpy(recv.copy()).cuda(), 2, chunk, out)
    torch.cuda.synchronize()
    got = to_host_u8(out)
    want = _reduce_expected(recv)
    bad = got != want
    assert not bad.any(), f"{int(bad.sum())} sums differ; first {np.argwhere(bad)[:5].ravel()}"
    # eight ranks of the largest code saturate; eight of the smallest subnormal stay exact
    recv8 = np.zeros((8, 16), np.uint8)
    recv8[:, 0] = 0x7B
    recv8[:, 1] = 0x01
    recv8[:, 2] = 0xFB
    out8 = torch.empty(16, dtype=torch.uint8, device="cuda")
    fp8.fp8_grad_reduce(torch.from_numpy(recv8).cuda(), 8, 16, out8)
    torch.cuda.synchronize()
    assert np.array_equal(to_host_u8(out8), _reduce_expected(recv8))
    assert to_host_u8(out8)[0] == 0x7B and to_host_u8(out8)[2] == 0xFB


@pytest.mark.parametrize("world", [12, 100, 128, 129, 300])
def test_reduce_kernel_wide_worlds(gpu_lib, world):
    """128 ranks: the fp32 path at its exactness limits (every rank at the
    largest code; sums of many subnormals, of mixed signs and magnitudes).
    12 and 100: the fp32 path's batches of eight ranks with a partial last
    batch.  More than 128: the integer path."""
    fp8 = gpu_lib
    rng = np.random.default_rng(world)
    finite = np.array([c for c in range(256) if (c & 0x7C) != 0x7C], dtype=np.uint8)
    chunk = 4096
    recv = rng.choice(finite, (world, chunk)).astype(np.uint8)
    recv[:, 0] = 0x7B                                   # world * 57344
    recv[:, 1] = 0x01                                   # world * 2^-16
    recv[:, 2] = np.where(np.arange(world) % 2, 0x03, 0x83)
    recv[:, 3] = 0x80                                   # all -0
    recv[:, 4:1000] = rng.choice(finite[(finite & 0x7C) < 0x14], (world, 996))  # small magnitudes only
    recv[:, 1000:2000] = rng.choice(finite[(finite & 0x7C) > 0x60], (world, 1000))  # large only
    out = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    fp8.fp8_grad_reduce(torch.from_numpy(recv).cuda(), world, chunk, out)
    torch.cuda.synchronize()
    got = to_host_u8(out)
    want = _reduce_expected(recv)
    bad = got != want
    assert not bad.any(), f"{int(bad.sum())} sums differ; first {np.argwhere(bad)[:5].ravel()}"


def test_argument_checks(gpu_lib):
    fp8 = gpu_lib
    g = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    a = torch.zeros(1, dtype=torch.float32, device="cuda")
    c = torch.zeros(64, dtype=torch.uint8, device="cuda")
    s = torch.zeros(2, dtype=torch.float32, device="cuda")
    with pytest.raises(fp8.Fp8Error):
        fp8.fp8_grad_quantize(g, 64, a, 0, c, 64, s)  # world 0
    with pytest.raises(fp8.Fp8Error):
        fp8.fp8_grad_quantize(g, 64, a, 2, c, 32, s)  # padded_n < n
    with pytest.raises(fp8.Fp8Error):
        fp8.fp8_grad_reduce(c, 2, 24, c)  # chunk not a multiple of 16
