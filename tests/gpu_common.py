"""Shared helpers of the GPU parity tests: run the library on a workload and compare
selected (layer, batch, head) slices with the oracle."""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import torch

import fibattn_inputs as fi
import oracle
import static_fibonacci_offset_fibattn_b300 as fa

TOL = {"f32": 1e-5, "bf16": 2e-2}   # max-abs, outputs of the forward and backward
LSE_TOL = {"f32": 1e-5, "bf16": 1e-3}


def lib_schedule(sched: dict) -> fa.Schedule:
    return fa.Schedule(**sched)


def oracle_table(sched: dict, layer: int, W: int, T: int):
    kind = sched.get("kind", "fixed")
    kw = {}
    if kind == "fixed":
        kw["alpha"] = Fraction(*sched.get("alpha", (1, 1)))
    else:
        kw["alpha_min"] = Fraction(*sched.get("alpha_min", (1, 2)))
        kw["alpha_max"] = Fraction(*sched.get("alpha_max", (3, 2)))
        kw["coprime_c"] = sched.get("coprime_c", 7)
    return oracle.layer_table(sched.get("base", "fib"), kind, layer, sched.get("n_layers", 1), W,
                              T, sched.get("base_max", 0), **kw)


def sample_slices(B, H, per_layer):
    """Deterministic (b, h) picks: first, last, and evenly spread ones."""
    all_bh = [(b, h) for b in range(B) for h in range(H)]
    if per_layer >= len(all_bh):
        return all_bh
    idx = np.unique(np.linspace(0, len(all_bh) - 1, per_layer).round().astype(int))
    return [all_bh[i] for i in idx]


def f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def oracle_fwd_slices(inp, sched, W, layer0, picks, scale=None):
    """Oracle forward on picked slices: picks = [(l, b, h)]. Returns dict pick -> (o, lse)."""
    T = inp["q"].shape[-2]
    out = {}
    by_layer = {}
    for (l, b, h) in picks:
        by_layer.setdefault(l, []).append((b, h))
    for l, bhs in by_layer.items():
        tab = oracle_table(sched, layer0 + l, W, T)
        q = np.stack([f64(inp["q"][l, b, h]) for b, h in bhs])
        k = np.stack([f64(inp["k"][l, b, h]) for b, h in bhs])
        v = np.stack([f64(inp["v"][l, b, h]) for b, h in bhs])
        o, lse = oracle.fwd(q, k, v, W, tab, scale)
        for n, (b, h) in enumerate(bhs):
            out[(l, b, h)] = (o[n], lse[n])
    return out


def oracle_bwd_slices(inp, sched, W, layer0, picks, scale=None):
    T = inp["q"].shape[-2]
    out = {}
    by_layer = {}
    for (l, b, h) in picks:
        by_layer.setdefault(l, []).append((b, h))
    for l, bhs in by_layer.items():
        tab = oracle_table(sched, layer0 + l, W, T)
        g = lambda n: np.stack([f64(inp[n][l, b, h]) for b, h in bhs])
        dq, dk, dv, o, lse = oracle.bwd(g("q"), g("k"), g("v"), g("dO"), W, tab, scale)
        for n, (b, h) in enumerate(bhs):
            out[(l, b, h)] = (dq[n], dk[n], dv[n], o[n], lse[n])
    return out


def to_dev(inp, device="cuda"):
    return {n: t.to(device) for n, t in inp.items()}


def max_abs(a, b):
    return float(np.max(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64))))


# Gradients are also gated relative to their own magnitude. The absolute bound alone cannot
# fail where gradients are small: on the training-step workload (inputs N(0,1)/8) the largest
# |dq| and |dk| of a slice are about 4e-3, a fifth of the bf16 bound, so an all-zero dq would
# pass it. The relative bound is 2e-2 of the tensor's largest reference magnitude on the bf16
# path (bf16 outputs carry 2^-9 relative rounding, and P, dS enter the products as bf16) and
# 1e-3 on the fp32 path; the small absolute floor admits gradients that vanish identically
# (a single query: dS = P (dO.v - dO.o) = 0), which the kernels reproduce only to rounding.
REL_TOL = {"f32": 1e-3, "bf16": 2e-2}
REL_FLOOR = {"f32": 1e-7, "bf16": 1e-6}


def grad_gate(got, ref, dtype):
    """(ok, err, rel): max-abs error within TOL[dtype] and within REL_TOL[dtype] of the
    largest |ref| (plus REL_FLOOR); rel = err / max |ref|."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = max_abs(got, ref)
    mag = float(np.max(np.abs(ref))) if ref.size else 0.0
    ok = err <= TOL[dtype] and err <= REL_TOL[dtype] * mag + REL_FLOOR[dtype]
    return ok, err, (err / mag if mag > 0 else 0.0)


def assert_grad(name, got, ref, dtype, where=""):
    ok, err, rel = grad_gate(got, ref, dtype)
    assert ok, (name, where, f"max-abs {err:.3g}", f"relative to max|ref| {rel:.3g}")
    return err, rel
