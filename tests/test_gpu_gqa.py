"""GPU parity of grouped-query (GQA / MQA) calls against the oracle.

Query head h reads kv head h // (H / H_kv); dk, dv of a kv row sum over the heads that read
it. Tolerances as the multi-head path (max-abs 1e-5 fp32, 2e-2 bf16; lse 1e-5 / 1e-3).
"""
import numpy as np
import pytest
import torch

import fibattn_inputs as fi
import oracle
import static_fibonacci_offset_fibattn_b300 as fa
from gpu_common import LSE_TOL, TOL, assert_grad, f64, lib_schedule, max_abs, oracle_table, to_dev

pytestmark = pytest.mark.gpu

SCHED = dict(kind="linear", base="fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=16)

GQA_EDGE = [
    # (Lc, B, H, Hkv, T, W)
    (1, 1, 8, 2, 300, 16),
    (1, 2, 8, 1, 257, 64),     # MQA, ragged last tile
    (2, 1, 6, 3, 129, 8),
    (1, 1, 4, 4, 200, 12),     # one kv head per query head
    (1, 1, 4, 2, 1, 4),
    (1, 1, 2, 1, 1100, 100),
]


def _inputs(Lc, B, H, Hkv, T, dtype, seed):
    kv = {n: (Lc, B, Hkv, T, 64) for n in ("k", "v")}
    return fi.draw((Lc, B, H, T, 64), seed=seed, scale=0.5, dtype=dtype,
                   names=("q", "k", "v", "dO"), shapes=kv)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", GQA_EDGE)
def test_gqa_fwd_bwd_matches_oracle(dtype, case):
    Lc, B, H, Hkv, T, W = case
    layer0 = 3
    inp = _inputs(Lc, B, H, Hkv, T, dtype, 100 + T)
    dev = to_dev(inp)
    sc = lib_schedule(SCHED)
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], W, sc, layer0=layer0)
    dq, dk, dv = fa.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["dO"], W, sc, layer0=layer0)
    torch.cuda.synchronize()
    fa.poll_device_error()
    assert dk.shape == dev["k"].shape and dv.shape == dev["v"].shape
    tabs = [oracle_table(SCHED, layer0 + l, W, T) for l in range(Lc)]
    g = lambda n: f64(inp[n])
    rq, rk, rv, ro, rl = oracle.bwd_gqa(g("q"), g("k"), g("v"), g("dO"), W, tabs)
    assert max_abs(f64(o), ro) <= TOL[dtype]
    assert max_abs(f64(lse), rl) <= LSE_TOL[dtype]
    for n, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert_grad(n, f64(got), ref, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gqa_equals_multi_head_on_repeated_kv(dtype):
    Lc, B, H, Hkv, T, W = 2, 2, 8, 2, 700, 64
    dev = to_dev(_inputs(Lc, B, H, Hkv, T, dtype, 7))
    sc = lib_schedule(SCHED)
    G = H // Hkv
    kr = dev["k"].repeat_interleave(G, dim=-3).contiguous()
    vr = dev["v"].repeat_interleave(G, dim=-3).contiguous()
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], W, sc)
    o2, lse2 = fa.fwd(dev["q"], kr, vr, W, sc)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    dq, dk, dv = fa.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["dO"], W, sc)
    dq2, dk2, dv2 = fa.bwd(dev["q"], kr, vr, o, lse, dev["dO"], W, sc)
    assert torch.equal(dq, dq2)
    shp = dk.shape[:-3] + (Hkv, G) + dk.shape[-2:]
    tol = 1e-5 if dtype == "f32" else 2e-2
    assert max_abs(f64(dk), f64(dk2.float().reshape(shp).sum(-3))) <= tol
    assert max_abs(f64(dv), f64(dv2.float().reshape(shp).sum(-3))) <= tol


def test_gqa_training_step_sampled():
    spec = fi.WORKLOADS["c5g"]
    inp = fi.workload_inputs("c5g")
    dev = to_dev(inp)
    sc = lib_schedule(spec["sched"])
    W = spec["W"]
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], W, sc)
    dq, dk, dv = fa.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["dO"], W, sc)
    torch.cuda.synchronize()
    fa.poll_device_error()
    G = spec["H"] // spec["Hkv"]
    # every layer: batch 0 and batch B-1, one kv head each (all the query heads that read it)
    for l in range(spec["Lc"]):
        tab = oracle_table(spec["sched"], l, W, spec["T"])
        for b in (0, spec["B"] - 1):
            hk = (l + b) % spec["Hkv"]
            hs = slice(hk * G, (hk + 1) * G)
            g = lambda n, hsl: f64(inp[n][l, b, hsl])[None]
            rq, rk, rv, ro, rl = oracle.bwd_gqa(g("q", hs), g("k", slice(hk, hk + 1)),
                                                g("v", slice(hk, hk + 1)), g("dO", hs), W, tab)
            assert max_abs(f64(o[l, b, hs])[None], ro) <= TOL["bf16"], (l, b)
            assert_grad("dq", f64(dq[l, b, hs])[None], rq, "bf16", (l, b))
            assert_grad("dk", f64(dk[l, b, hk:hk + 1])[None], rk, "bf16", (l, b))
            assert_grad("dv", f64(dv[l, b, hk:hk + 1])[None], rv, "bf16", (l, b))


def test_gqa_autograd_wrapper():
    dev = to_dev(_inputs(1, 1, 4, 1, 300, "bf16", 9))
    sc = lib_schedule(SCHED)
    q, k, v = (dev[n][0].clone().requires_grad_(True) for n in ("q", "k", "v"))
    o = fa.FibSparseAttention.apply(q, k, v, 16, sc)
    o.backward(dev["dO"][0])
    o2, lse = fa.fwd(dev["q"][0], dev["k"][0], dev["v"][0], 16, sc)
    g = fa.bwd(dev["q"][0], dev["k"][0], dev["v"][0], o2, lse, dev["dO"][0], 16, sc)
    assert torch.equal(q.grad, g[0]) and torch.equal(k.grad, g[1]) and torch.equal(v.grad, g[2])


def test_gqa_rejects_bad_head_counts():
    q = torch.zeros(1, 6, 64, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 4, 64, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        fa.fwd(q, k, k, 8, lib_schedule(SCHED))
