"""The FP8 gradient all-reduce's host logic on CPU ranks (gloo): chunking,
padding, the MAX all-reduce of the amax, the all-to-all of codes and the
all-gather of the reduced chunks (grad_allreduce.all_reduce).

The device steps are injected: each is restated here with the oracle's
primitives (amax, scale rule, cast, decode, exact sum, encode), on CPU
tensors.  The result of the distributed decomposition must equal, bit for
bit, the oracle's all-reduce computed on all ranks' gradients at once."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle


class OracleOps:
    """fp8_grad_* restated with the oracle, on CPU tensors."""

    def amax(self, g):
        return torch.tensor([float(oracle.amax(_bits(g)))], dtype=torch.float32)

    def quantize(self, g, amax, world, padded_n):
        s = oracle.allreduce_scale(float(amax[0]), world)
        q, _, _ = oracle.cast(_bits(g), s, oracle.E5M2)
        codes = torch.zeros(padded_n, dtype=torch.uint8)
        codes[:q.size] = torch.from_numpy(q)
        return codes, torch.tensor([s, oracle.reciprocal(s)], dtype=torch.float32)

    def reduce(self, recv, world, chunk):
        dec = oracle.decode(recv.numpy().reshape(world, chunk), oracle.E5M2)
        total = dec[0].copy()
        for r in range(1, world):
            total = total + dec[r]  # exact; keeps -0 + -0 = -0
        return torch.tensor([oracle.encode_double(v, oracle.E5M2) for v in total], dtype=torch.uint8)

    def dequantize(self, codes, n, scale, world, average):
        f = np.float32(scale[1].item())
        if average:
            f = np.float32(f / np.float32(world))
        y = (oracle.decode(codes.numpy()[:n], oracle.E5M2).astype(np.float32) * f).astype(np.float32)
        return torch.from_numpy(oracle.f64_to_bf16(y.astype(np.float64)).view(np.int16)).view(torch.bfloat16)


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _grad(rank, n, seed):
    from fp8_mixed_precision_history_gb300 import synthetic

    return synthetic.grad_like((n,), seed + 17 * rank)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, n, seed, average, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from fp8_mixed_precision_history_gb300 import grad_allreduce

        g = _grad(rank, n, seed)
        out = grad_allreduce.all_reduce(g, average=average, ops=OracleOps())
        want, _, _ = oracle.allreduce_e5m2(np.stack([_bits(_grad(r, n, seed)) for r in range(world)]),
                                           average=average)
        q.put((rank, bool(np.array_equal(_bits(out), want)), int(np.count_nonzero(_bits(out) != want))))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,n,average", [(2, 1000, False), (2, 4099, True), (3, 777, False)])
def test_gloo_all_reduce_matches_oracle(world, n, average):
    oracle.lib()  # build once, before the workers start
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, n, 40 + n, average, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, ok, bad in out:
        assert ok, f"rank {rank}: {bad} elements differ from the oracle"


def test_chunking():
    from fp8_mixed_precision_history_gb300.grad_allreduce import chunk_size

    assert chunk_size(1, 1) == 16
    assert chunk_size(1000, 2) == 512
    assert chunk_size(4099, 2) == 2064
    assert chunk_size(777, 3) == 272
    for n in (1, 15, 16, 17, 1000, 65536 * 3 + 7):
        for w in (1, 2, 3, 8):
            c = chunk_size(n, w)
            assert c % 16 == 0 and c * w >= n and (c - 16) * w < n


def test_local_emulation_matches_oracle_on_cpu():
    """all_reduce_local (several ranks in one process) with the oracle ops."""
    from fp8_mixed_precision_history_gb300 import grad_allreduce

    grads = [_grad(r, 333, 5) for r in range(4)]
    out, codes = grad_allreduce.all_reduce_local(grads, average=True, ops=OracleOps(), with_codes=True)
    want, wcodes, _ = oracle.allreduce_e5m2(np.stack([_bits(g) for g in grads]), average=True)
    assert np.array_equal(_bits(out), want)
    assert np.array_equal(codes.numpy(), wcodes)
