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


def bits(t):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def codes(t):
    """uint8 tensor -> numpy uint8 (host copy)."""
    return t.detach().cpu().contiguous().numpy()
