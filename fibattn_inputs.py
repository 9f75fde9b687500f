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


def draw(shape, seed: int, scale: float, dtype: str = "bf16", names=("q", "k", "v"), shapes=None):
    """Return a dict name -> CPU tensor of `shape` (or shapes[name]), drawn in `names` order."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    out = {}
    for name in names:
        shp = (shapes or {}).get(name, shape)
        x = torch.randn(tuple(shp), generator=g, dtype=torch.float32) * float(scale)
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


# Workloads shaped like the pages' model (hidden 512 = 8 heads x 64, 16 layers,
# trained length 1024 and 4x = 4096). Plain data: shapes, seeds, scales, schedules.
# 'sched' keys follow the library's Schedule fields; 'seed' is an int (one draw shared
# by every layer, stored in distinct per-layer buffers) or 'per_layer:<s0>' (seed s0 + l).
WORKLOADS = {
    "c1": dict(desc="single sparse-attention layer, fp32", dtype="f32", Lc=1, B=1, H=2, T=256,
               d=64, W=16, seed=0, scale=1.0, names=("q", "k", "v"), passes=("fwd",),
               sched=dict(kind="fixed", base="fib", alpha=(1, 1), n_layers=1)),
    "c2": dict(desc="one layer of the 60M model, bf16", dtype="bf16", Lc=1, B=8, H=8, T=1024,
               d=64, W=64, seed=1, scale=0.125, names=("q", "k", "v"), passes=("fwd",),
               sched=dict(kind="fixed", base="fib", alpha=(1, 1), n_layers=1)),
    "c3": dict(desc="16-layer stack, linear stagger 0.5->2.0, bf16", dtype="bf16", Lc=16, B=8,
               H=8, T=1024, d=64, W=64, seed="per_layer:2", scale=0.125, names=("q", "k", "v"),
               passes=("fwd",),
               sched=dict(kind="linear", base="fib", alpha_min=(1, 2), alpha_max=(2, 1),
                          n_layers=16)),
    "c3p": dict(desc="16-layer stack, power-of-two control (alpha = 1), bf16", dtype="bf16",
                Lc=16, B=8, H=8, T=1024, d=64, W=64, seed="per_layer:2", scale=0.125,
                names=("q", "k", "v"), passes=("fwd",),
                sched=dict(kind="fixed", base="pow2", alpha=(1, 1), n_layers=16)),
    "c4": dict(desc="4x length extrapolation, 16 layers, linear stagger 0.5->2.0, bf16",
               dtype="bf16", Lc=16, B=2, H=8, T=4096, d=64, W=64, seed=3, scale=0.125,
               names=("q", "k", "v"), passes=("fwd",),
               sched=dict(kind="linear", base="fib", alpha_min=(1, 2), alpha_max=(2, 1),
                          n_layers=16)),
    "c5": dict(desc="training step fwd+bwd, 16 layers, coprime (5l mod 16) of the linear "
                    "stagger 0.5->2.0, bf16", dtype="bf16", Lc=16, B=8, H=8, T=1024, d=64,
               W=64, seed=4, scale=0.125, names=("q", "k", "v", "dO"), passes=("fwd", "bwd"),
               sched=dict(kind="coprime", base="fib", alpha_min=(1, 2), alpha_max=(2, 1),
                          n_layers=16, coprime_c=5)),
    "c5o": dict(desc="training step fwd+bwd with the one-pass backward (a thread block per tile "
                     "owns dq of its queries and dk, dv of its keys), 16 layers, coprime (5l mod 16) "
                     "of the linear stagger 0.5->2.0, bf16", dtype="bf16", Lc=16, B=8, H=8, T=1024,
                d=64, W=64, seed=4, scale=0.125, names=("q", "k", "v", "dO"),
                passes=("fwd", "bwd"), bwd_fused=True,
                sched=dict(kind="coprime", base="fib", alpha_min=(1, 2), alpha_max=(2, 1),
                           n_layers=16, coprime_c=5)),
    "c5g": dict(desc="training step fwd+bwd, 16 layers, grouped-query (8 query heads sharing 2 "
                     "kv heads), coprime (5l mod 16) of the linear stagger 0.5->2.0, bf16",
                dtype="bf16", Lc=16, B=8, H=8, Hkv=2, T=1024, d=64, W=64, seed=4, scale=0.125,
                names=("q", "k", "v", "dO"), passes=("fwd", "bwd"),
                sched=dict(kind="coprime", base="fib", alpha_min=(1, 2), alpha_max=(2, 1),
                           n_layers=16, coprime_c=5)),
    "c5r": dict(desc="training step fwd+bwd with RoPE on q and k before the gather (base 10000), "
                     "16 layers, coprime (5l mod 16) of the linear stagger 0.5->2.0, bf16",
                dtype="bf16", Lc=16, B=8, H=8, T=1024, d=64, W=64, seed=4, scale=0.125,
                names=("q", "k", "v", "dO"), passes=("fwd", "bwd"), rope_base=10000.0,
                sched=dict(kind="coprime", base="fib", alpha_min=(1, 2), alpha_max=(2, 1),
                           n_layers=16, coprime_c=5)),
    "c3r": dict(desc="16-layer stack forward with RoPE on q and k (base 10000) applied inside "
                     "the attention kernel (no rotated copies), linear stagger 0.5->2.0, bf16",
                dtype="bf16", Lc=16, B=8, H=8, T=1024, d=64, W=64, seed="per_layer:2", scale=0.125,
                names=("q", "k", "v"), passes=("fwd",), rope_base=10000.0, rope_fused=True,
                sched=dict(kind="linear", base="fib", alpha_min=(1, 2), alpha_max=(2, 1),
                           n_layers=16)),
    "c3w": dict(desc="16-layer stack at head size 128 (4 heads x 128 = the same hidden 512), "
                     "linear stagger 0.5->2.0, bf16", dtype="bf16", Lc=16, B=8, H=4, T=1024, d=128,
                W=64, seed="per_layer:2", scale=0.125, names=("q", "k", "v"), passes=("fwd",),
                sched=dict(kind="linear", base="fib", alpha_min=(1, 2), alpha_max=(2, 1),
                           n_layers=16)),
    "c5w": dict(desc="training step fwd+bwd at head size 128 (4 heads x 128), coprime (5l mod 16) "
                     "of the linear stagger 0.5->2.0, bf16", dtype="bf16", Lc=16, B=8, H=4, T=1024,
                d=128, W=64, seed=4, scale=0.125, names=("q", "k", "v", "dO"),
                passes=("fwd", "bwd"),
                sched=dict(kind="coprime", base="fib", alpha_min=(1, 2), alpha_max=(2, 1),
                           n_layers=16, coprime_c=5)),
    "c3f": dict(desc="16-layer stack, fractional (learned-style) alphas in [0.5, 2.0], bf16",
                dtype="bf16", Lc=16, B=8, H=8, T=1024, d=64, W=64, seed="per_layer:2",
                scale=0.125, names=("q", "k", "v"), passes=("fwd",), base="fib",
                alphas=dict(lo=0.5, hi=2.0, seed=7)),
    "c5f": dict(desc="training step fwd+bwd (with dL/dalpha), 16 layers, fractional "
                     "(learned-style) alphas in [0.5, 2.0], bf16", dtype="bf16", Lc=16, B=8, H=8,
                T=1024, d=64, W=64, seed=4, scale=0.125, names=("q", "k", "v", "dO"),
                passes=("fwd", "bwd"), base="fib", alphas=dict(lo=0.5, hi=2.0, seed=7)),
}


def frac_alphas(spec):
    """Per-layer float32 alphas of a fractional-offset workload: Lc uniform draws in
    [lo, hi) from their own generator, sorted ascending (deeper layers reach further, as
    in a stagger). Returns a list of Python floats holding float32 values."""
    a = spec["alphas"]
    g = torch.Generator("cpu").manual_seed(int(a["seed"]))
    x = torch.rand(spec["Lc"], generator=g, dtype=torch.float32) * (a["hi"] - a["lo"]) + a["lo"]
    return [float(v) for v in torch.sort(x).values]


def seed_of(spec):
    s = spec["seed"]
    if isinstance(s, str) and s.startswith("per_layer:"):
        s0 = int(s.split(":")[1])
        return lambda l: s0 + l
    return int(s)


def workload_inputs(name: str, layers=None, **override):
    """CPU tensors [Lc, B, H, T, d] of a named workload (optionally only `layers`)."""
    spec = dict(WORKLOADS[name], **override)
    shape = (spec["B"], spec["H"], spec["T"], spec["d"])
    # grouped-query workloads: k and v have Hkv heads
    kv = {n: (spec["B"], spec["Hkv"], spec["T"], spec["d"]) for n in ("k", "v")} if "Hkv" in spec else None
    seed = seed_of(spec)
    Lc = spec["Lc"]
    if layers is None:
        layers = list(range(Lc))
    if callable(seed):
        per = [draw(shape, seed(l), spec["scale"], spec["dtype"], spec["names"], kv) for l in layers]
    else:
        one = draw(shape, seed, spec["scale"], spec["dtype"], spec["names"], kv)
        per = [{n: t.clone() for n, t in one.items()} for _ in layers]
    return {n: torch.stack([p[n] for p in per]).contiguous() for n in spec["names"]}
