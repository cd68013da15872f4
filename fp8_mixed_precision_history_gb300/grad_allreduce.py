"""FP8 (E5M2) gradient all-reduce with automatic scaling.

"FP8 and low-precision formats" (aiunderstanding.org), use cases: E5M2 for
gradient communication in distributed training, to cut inter-node bandwidth.
"[📪정보] 그저께 나온 논문 대박이네" (mir.rootios.com, a thread on the FP8-LM paper):
automatic scaling adjusts the tensor scaling factor so that gradients stay
inside FP8's range during the all-reduce.

Every arithmetic step runs in the library's kernels (``fp8_grad_amax``,
``fp8_grad_quantize``, ``fp8_grad_reduce``, ``fp8_grad_dequantize``; see
include/fp8lin.h).  This module only chooses the chunking, allocates buffers
and moves bytes between ranks:

1. local amax, then a MAX all-reduce of one float: the shared amax;
2. codes = E5M2(g * s), s = 57344 / (world * amax), padded to world * chunk;
3. all-to-all: rank r receives chunk r of every rank's codes;
4. exact sum of the world chunks, rounded once to E5M2;
5. all-gather of the reduced chunks;
6. bf16(decode(code) * 1/s), or the mean.

One byte per element crosses the network in each of steps 3 and 5.
"""
import torch

CHUNK_ALIGN = 16  # bytes: the reduce kernel reads 16 codes per thread


def chunk_size(n, world):
    """Codes per rank chunk: ceil(n / world) rounded up to a multiple of 16."""
    c = -(-n // world)
    return CHUNK_ALIGN * max(1, -(-c // CHUNK_ALIGN))


class LibraryOps:
    """The four device steps as the CUDA library runs them (device tensors)."""

    def __init__(self, stream=None):
        import fp8_mixed_precision_history_gb300 as fp8

        self.fp8 = fp8
        self.stream = stream

    def amax(self, g):
        a = torch.empty(1, dtype=torch.float32, device=g.device)
        self.fp8.fp8_grad_amax(g, g.numel(), a, self.stream)
        return a

    def quantize(self, g, amax, world, padded_n):
        codes = torch.empty(padded_n, dtype=torch.uint8, device=g.device)
        scale = torch.empty(2, dtype=torch.float32, device=g.device)
        self.fp8.fp8_grad_quantize(g, g.numel(), amax, world, codes, padded_n, scale, self.stream)
        return codes, scale

    def reduce(self, recv, world, chunk):
        out = torch.empty(chunk, dtype=torch.uint8, device=recv.device)
        self.fp8.fp8_grad_reduce(recv, world, chunk, out, self.stream)
        return out

    def dequantize(self, codes, n, scale, world, average):
        out = torch.empty(n, dtype=torch.bfloat16, device=codes.device)
        self.fp8.fp8_grad_dequantize(codes, n, scale, world, average, out, self.stream)
        return out


def all_reduce(grad, group=None, average=False, ops=None):
    """All-reduce a bf16 gradient over the ranks of a torch.distributed group
    through E5M2 codes.  Returns a new bf16 tensor of grad's shape holding the
    sum (or the mean, ``average=True``), the same on every rank."""
    import torch.distributed as dist

    ops = ops or LibraryOps()
    world = dist.get_world_size(group)
    flat = grad.contiguous().view(-1)
    n = flat.numel()
    chunk = chunk_size(n, world)
    padded = chunk * world
    amax = ops.amax(flat)
    dist.all_reduce(amax, op=dist.ReduceOp.MAX, group=group)
    codes, scale = ops.quantize(flat, amax, world, padded)
    recv = torch.empty_like(codes)
    dist.all_to_all_single(recv, codes, group=group)
    mine = ops.reduce(recv, world, chunk)
    full = torch.empty(padded, dtype=torch.uint8, device=codes.device)
    dist.all_gather_into_tensor(full, mine, group=group)
    return ops.dequantize(full, n, scale, world, average).view(grad.shape)


def all_reduce_local(grads, average=False, ops=None, with_codes=False):
    """The same all-reduce for len(grads) ranks emulated in one process (for
    example on one GPU): each rank's steps run in turn and the exchanges are
    plain device copies -- no kernel waits on another.  Returns the result
    every rank would hold (and, with ``with_codes``, the reduced codes)."""
    ops = ops or LibraryOps()
    world = len(grads)
    flats = [g.contiguous().view(-1) for g in grads]
    n = flats[0].numel()
    assert all(f.numel() == n for f in flats)
    chunk = chunk_size(n, world)
    padded = chunk * world
    amax = torch.stack([ops.amax(f) for f in flats]).max().reshape(1)  # stands in for the MAX all-reduce
    quant = [ops.quantize(f, amax, world, padded) for f in flats]
    reduced = []
    for r in range(world):
        recv = torch.cat([quant[j][0][r * chunk:(r + 1) * chunk] for j in range(world)])
        reduced.append(ops.reduce(recv, world, chunk))
    full = torch.cat(reduced)
    out = ops.dequantize(full, n, quant[0][1], world, average).view(grads[0].shape)
    return (out, full[:n]) if with_codes else out
