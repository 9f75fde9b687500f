"""GPU parity of the rotary position embedding kernels and of the attention through them.

The table (fp64 cos/sin rounded once to float32) must agree with fp64 to one float ulp; the
rotation within the output dtype's rounding; the attention through RoPE within the path's
tolerances (max-abs 1e-5 fp32, 2e-2 bf16; lse 1e-5 / 1e-3).
"""
import numpy as np
import pytest
import torch

import fibattn_inputs as fi
import oracle
import static_fibonacci_offset_fibattn_b300 as fa
from gpu_common import LSE_TOL, TOL, assert_grad, f64, lib_schedule, max_abs, oracle_table, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,base", [(1, 10000.0), (1024, 10000.0), (4096, 10000.0), (300, 500.0)])
def test_rope_table_matches_fp64(T, base):
    t = fa.rope_table(T, base).cpu().numpy().astype(np.float64)
    theta = base ** (-2.0 * np.arange(32) / 64)
    ang = np.arange(T)[:, None] * theta[None, :]
    ref = np.stack((np.cos(ang), np.sin(ang)), axis=-1)
    assert np.all(np.abs(t - ref) <= 2.0 ** -24 * np.abs(ref) + 1e-30)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", [(3, 257, 64), (2, 2, 1024, 64), (1, 1, 64)])
@pytest.mark.parametrize("inverse", [False, True])
def test_rope_kernel_matches_oracle(dtype, shape, inverse):
    x = fi.draw(shape, seed=5, scale=2.0, dtype=dtype, names=("x",))["x"]
    T = shape[-2]
    table = fa.rope_table(T)
    y = fa.rope(x.cuda(), table, inverse=inverse)
    ref = oracle.rope(f64(x), inverse=inverse)
    if dtype == "f32":
        assert max_abs(f64(y), ref) <= 2e-6
    else:  # one bf16 rounding of the result
        assert np.all(np.abs(f64(y) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)


def test_rope_in_place_and_round_trip():
    x = fi.draw((2, 3, 500, 64), seed=6, scale=1.0, dtype="f32", names=("x",))["x"].cuda()
    table = fa.rope_table(500)
    y = fa.rope(x, table)
    z = x.clone()
    fa.rope(z, table, out=z)
    assert torch.equal(y, z)
    back = fa.rope(y, table, inverse=True)
    assert max_abs(f64(back), f64(x)) <= 2e-6
    with pytest.raises(ValueError):
        fa.rope(x, fa.rope_table(100))  # table shorter than T


SCHED = dict(kind="linear", base="fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=16)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", [(1, 2, 2, 300, 16), (2, 4, 1, 1030, 64), (1, 8, 2, 257, 8)])
def test_attention_through_rope_matches_oracle(dtype, case):
    Lc, H, Hkv, T, W = case
    kv = {n: (Lc, 1, Hkv, T, 64) for n in ("k", "v")}
    inp = fi.draw((Lc, 1, H, T, 64), seed=T, scale=0.5, dtype=dtype, names=("q", "k", "v", "dO"),
                  shapes=kv)
    dev = to_dev(inp)
    sc = lib_schedule(SCHED)
    table = fa.rope_table(T)
    o, lse, (qr, kr) = fa.fwd_rope(dev["q"], dev["k"], dev["v"], W, sc, table, layer0=5)
    dq, dk, dv = fa.bwd_rope(qr, kr, dev["v"], o, lse, dev["dO"], W, sc, table, layer0=5)
    torch.cuda.synchronize()
    fa.poll_device_error()
    tabs = [oracle_table(SCHED, 5 + l, W, T) for l in range(Lc)]
    g = lambda n: f64(inp[n])
    rq, rk, rv, ro, rl = oracle.bwd_rope(g("q"), g("k"), g("v"), g("dO"), W, tabs)
    assert max_abs(f64(o), ro) <= TOL[dtype]
    assert max_abs(f64(lse), rl) <= LSE_TOL[dtype]
    for n, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert_grad(n, f64(got), ref, dtype)


def test_rope_training_step_sampled():
    spec = fi.WORKLOADS["c5r"]
    inp = fi.workload_inputs("c5r")
    dev = to_dev(inp)
    sc = lib_schedule(spec["sched"])
    W, T = spec["W"], spec["T"]
    table = fa.rope_table(T, spec["rope_base"])
    o, lse, (qr, kr) = fa.fwd_rope(dev["q"], dev["k"], dev["v"], W, sc, table)
    dq, dk, dv = fa.bwd_rope(qr, kr, dev["v"], o, lse, dev["dO"], W, sc, table)
    torch.cuda.synchronize()
    fa.poll_device_error()
    for l in (0, 7, 15):
        tab = oracle_table(spec["sched"], l, W, T)
        b, h = l % spec["B"], (3 * l) % spec["H"]
        g = lambda n: f64(inp[n][l, b, h])[None]
        rq, rk, rv, ro, rl = oracle.bwd_rope(g("q"), g("k"), g("v"), g("dO"), W, tab,
                                             spec["rope_base"])
        assert max_abs(f64(o[l, b, h])[None], ro) <= TOL["bf16"], l
        for n, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
            assert_grad(n, f64(got[l, b, h])[None], ref, "bf16", l)


# ------------------------------------------------------------------ RoPE inside the forward

FUSED = [
    # (Lc, B, H, Hkv, T, W)
    (1, 1, 2, 2, 1, 4),
    (1, 1, 2, 1, 300, 16),
    (2, 1, 4, 2, 1030, 64),     # ragged last tile, grouped heads, two layers
    (1, 2, 2, 2, 257, 8),
    (1, 1, 2, 2, 700, 200),     # several band groups per tile
    (1, 1, 1, 1, 2049, 64),
]


@pytest.mark.parametrize("case", FUSED)
def test_fused_rope_forward_matches_oracle(case):
    # the oracle rotates in fp64 and attends over the rotated tensors (fwd_rope)
    Lc, B, H, Hkv, T, W = case
    kv = {n: (Lc, B, Hkv, T, 64) for n in ("k", "v")}
    inp = fi.draw((Lc, B, H, T, 64), seed=300 + T, scale=0.5, dtype="bf16", shapes=kv)
    dev = to_dev(inp)
    sc = lib_schedule(SCHED)
    table = fa.rope_table(T)
    o, lse = fa.fwd_rope_fused(dev["q"], dev["k"], dev["v"], W, sc, table, layer0=5)
    torch.cuda.synchronize()
    fa.poll_device_error()
    tabs = [oracle_table(SCHED, 5 + l, W, T) for l in range(Lc)]
    ro, rl = oracle.fwd_rope(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), W, tabs)
    assert max_abs(f64(o), ro) <= TOL["bf16"]
    assert max_abs(f64(lse), rl) <= LSE_TOL["bf16"]
    # and the unfused path (rotated copies, then the attention) to rounding
    o2, l2, _ = fa.fwd_rope(dev["q"], dev["k"], dev["v"], W, sc, table, layer0=5)
    assert max_abs(f64(o), f64(o2)) <= TOL["bf16"]
    assert max_abs(f64(lse), f64(l2)) <= LSE_TOL["bf16"]


def test_fused_rope_forward_training_shape_sampled():
    # the 16-layer training-step shape with RoPE, forward only, in one call
    spec = fi.WORKLOADS["c5r"]
    inp = fi.workload_inputs("c5r", names=("q", "k", "v"))
    dev = to_dev(inp)
    sc = lib_schedule(spec["sched"])
    W, T = spec["W"], spec["T"]
    table = fa.rope_table(T, spec["rope_base"])
    o, lse = fa.fwd_rope_fused(dev["q"], dev["k"], dev["v"], W, sc, table)
    torch.cuda.synchronize()
    fa.poll_device_error()
    for l in (0, 9, 15):
        tab = oracle_table(spec["sched"], l, W, T)
        b, h = (5 * l) % spec["B"], (l + 3) % spec["H"]
        g = lambda n: f64(inp[n][l, b, h])[None]
        ro, rl = oracle.fwd_rope(g("q"), g("k"), g("v"), W, tab, spec["rope_base"])
        assert max_abs(f64(o[l, b, h])[None], ro) <= TOL["bf16"], l
        assert max_abs(f64(lse[l, b, h])[None], rl) <= LSE_TOL["bf16"], l


def test_fused_rope_forward_deterministic_and_in_place_safe():
    inp = to_dev(fi.draw((2, 2, 2, 1024, 64), seed=17, scale=0.5, dtype="bf16"))
    sc = lib_schedule(SCHED)
    table = fa.rope_table(1024)
    q0, k0 = inp["q"].clone(), inp["k"].clone()
    a = fa.fwd_rope_fused(inp["q"], inp["k"], inp["v"], 64, sc, table)
    b = fa.fwd_rope_fused(inp["q"], inp["k"], inp["v"], 64, sc, table)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    # the inputs are read, never written (the rotation happens in shared memory)
    assert torch.equal(inp["q"], q0) and torch.equal(inp["k"], k0)
