"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module holds random-number plumbing only: it contains none of the attention
method's arithmetic, so both the CUDA path and the CPU oracle can be fed from it
without sharing any computation.

Recipe (one draw per tensor, in a fixed order):
    g = torch.Generator('cpu').manual_seed(seed)
    for name in names:                      # e.g. q, k, v[, dO]
        x = torch.randn(shape, generator=g, dtype=torch.float32) * scale
        x = x.to(dtype)                     # round once on the CPU
Both sides consume exactly the rounded values; the oracle upcasts them to fp64.
"""
from __future__ import annotations

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def draw(shape, seed: int, scale: float, dtype: str = "bf16", names=("q", "k", "v")):
    """Return a dict name -> CPU tensor of `shape`, drawn in `names` order."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    out = {}
    for name in names:
        x = torch.randn(tuple(shape), generator=g, dtype=torch.float32) * float(scale)
        out[name] = x.to(DTYPES[dtype]).contiguous()
    return out


def draw_layers(n_layers: int, slice_shape, seed, scale: float, dtype: str = "bf16",
                names=("q", "k", "v")):
    """Stack per-layer draws into [Lc, *slice_shape] tensors.

    `seed` is either an int (one draw, copied into every layer's buffer) or a
    callable layer -> seed (an independent draw per layer)."""
    per = []
    if callable(seed):
        for l in range(n_layers):
            per.append(draw(slice_shape, seed(l), scale, dtype, names))
    else:
        one = draw(slice_shape, seed, scale, dtype, names)
        per = [one] * n_layers
    return {n: torch.stack([p[n] for p in per]).contiguous() for n in names}


def to_f64(t: torch.Tensor):
    """Exact upcast of a (possibly bf16) CPU tensor to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()
