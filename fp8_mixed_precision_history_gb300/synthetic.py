"""Seeded synthetic inputs shaped like the pages' workloads.

This module draws random numbers and nothing else: it holds none of the FP8
method's arithmetic, so both the CUDA path and the CPU oracle can consume the
same tensors.  Every generator is a ``torch.Generator`` seeded explicitly;
values are drawn in fp32 and rounded once to bf16 (the inputs of the linear
layer are bf16 tensors).

Workloads ("4.2 Hopper I -- Transformer Engine / FP8", S4.2.6: a transformer
layer with hidden size 4096 and FFN size 16384):

* linear layers (in -> out): QKV 4096->12288, attention projection 4096->4096,
  FC1 4096->16384, FC2 16384->4096; weight W is [out, in] and Y = X . W^T.
* activations ~ N(0, 1), weights ~ N(0, 0.02).
* output gradients: random sign, magnitude log-uniform on [1e-6, 1e-1].
* the cast sweep: N(0, 1) with 0.1% of the positions (a seeded Bernoulli draw)
  multiplied by 100, and an all-small variant N(0, 1e-3).
"""
import math

import torch

HIDDEN = 4096
FFN = 16384
# (name, in_features, out_features)
TE_LAYERS = (
    ("qkv", HIDDEN, 3 * HIDDEN),
    ("proj", HIDDEN, HIDDEN),
    ("fc1", HIDDEN, FFN),
    ("fc2", FFN, HIDDEN),
)

KIND = {"x": 0, "w": 1, "dy": 2}


def seed_for(cfg, layer=0, kind="x", step=0):
    """Seed rule: 1000*cfg + 10*layer + {x:0, w:1, dy:2} + 100*step."""
    return 1000 * cfg + 10 * layer + KIND[kind] + 100 * step


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, std, seed, device="cpu"):
    """bf16 tensor of N(0, std^2) draws."""
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return (x * std).to(torch.bfloat16)


def spiky(shape, seed, frac=1e-3, mult=100.0, device="cpu"):
    """N(0, 1) with a seeded Bernoulli(frac) subset of positions scaled by mult.

    The positions come from a second generator seeded with seed + 50."""
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    g2 = _gen(seed + 50, device)
    u = torch.rand(shape, generator=g2, device=device, dtype=torch.float32)
    x = torch.where(u < frac, x * mult, x)
    return x.to(torch.bfloat16)


def grad_like(shape, seed, lo=1e-6, hi=1e-1, device="cpu"):
    """Random sign (p = 1/2) times exp(U(ln lo, ln hi))."""
    g = _gen(seed, device)
    u = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    s = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    mag = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    return torch.where(s < 0.5, -mag, mag).to(torch.bfloat16)


def single_linear(seed=0, tokens=256, in_features=512, out_features=512, std=0.02):
    """X [tokens, in] then W [out, in], both N(0, std^2), from ONE generator."""
    g = _gen(seed, "cpu")
    x = (torch.randn((tokens, in_features), generator=g) * std).to(torch.bfloat16)
    w = (torch.randn((out_features, in_features), generator=g) * std).to(torch.bfloat16)
    return x, w


def block_varied(shape, seed, span=24, zero_frac=0.02, device="cpu"):
    """N(0, 1) rows whose 32-element blocks (along the last axis) each carry
    their own magnitude 2^e, e uniform on [-span, span], and a seeded fraction
    of blocks set to zero -- inputs whose per-block scales differ.  A third of
    the blocks have their largest entry moved onto 1.75 * 2^e or the next bf16
    value above it, the two sides of the FP8_MAX boundary of a power-of-two
    block scale (E4M3 448 = 1.75 * 2^8, E5M2 57344 = 1.75 * 2^15)."""
    rows, cols = shape
    nb = (cols + 31) // 32
    g = _gen(seed, device)
    x = torch.randn((rows, nb * 32), generator=g, device=device, dtype=torch.float32)
    e = torch.randint(-span, span + 1, (rows, nb, 1), generator=g, device=device).to(torch.float32)
    z = torch.rand((rows, nb, 1), generator=g, device=device) < zero_frac
    edge = torch.randint(0, 3, (rows, nb), generator=g, device=device)
    x = x.view(rows, nb, 32) / 4.0  # |x| < 1.75 in almost every block
    pos = torch.randint(0, 32, (rows, nb, 1), generator=g, device=device)
    top = torch.where(edge == 1, torch.full_like(e[..., 0], 1.75), torch.full_like(e[..., 0], 1.7578125))
    x = torch.where(((edge > 0).unsqueeze(-1)) & (torch.arange(32, device=device) == pos),
                    top.unsqueeze(-1), x)
    x = x * torch.exp2(e)
    x = torch.where(z, torch.zeros_like(x), x)
    return x.reshape(rows, nb * 32)[:, :cols].to(torch.bfloat16).contiguous()


def bits(t):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def codes(t):
    """uint8 tensor -> numpy uint8 (host copy)."""
    return t.detach().cpu().contiguous().numpy()
