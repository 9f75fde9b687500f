"""GPU parity of the fractional-offset (learned-alpha) forward against the oracle.

Values within the stated max-abs tolerances (1e-5 fp32 path, 2e-2 bf16 path; lse 1e-5 /
1e-3); an integer alpha must reproduce the static kernels bit for bit; the full 16-layer
workload runs in the configuration the benchmark times, with sampled slices recomputed
by the oracle.
"""
import numpy as np
import pytest
import torch

import fibattn_inputs as fi
import oracle
import static_fibonacci_offset_fibattn_b300 as fa
from gpu_common import LSE_TOL, TOL, assert_grad, f64, max_abs, sample_slices, to_dev

pytestmark = pytest.mark.gpu


def f32(a):
    return float(np.float32(a))


def oracle_frac_slices(inp, alphas, base, W, picks, scale=None):
    T = inp["q"].shape[-2]
    out, by_layer = {}, {}
    for (l, b, h) in picks:
        by_layer.setdefault(l, []).append((b, h))
    for l, bhs in by_layer.items():
        dists = oracle.frac_distances(f32(alphas[l]), base, W, T)
        g = lambda n: np.stack([f64(inp[n][l, b, h]) for b, h in bhs])
        o, lse = oracle.fwd_frac(g("q"), g("k"), g("v"), W, dists, scale)
        for n, (b, h) in enumerate(bhs):
            out[(l, b, h)] = (o[n], lse[n])
    return out


def test_fwd_frac_c3f_sixteen_layers_sampled():
    spec = fi.WORKLOADS["c3f"]
    alphas = fi.frac_alphas(spec)
    inp = fi.workload_inputs("c3f")
    dev = to_dev(inp)
    o, lse = fa.fwd_frac(dev["q"], dev["k"], dev["v"], spec["W"], alphas, spec["base"])
    torch.cuda.synchronize()
    fa.poll_device_error()
    picks = [(l, b, h) for l in range(spec["Lc"]) for (b, h) in sample_slices(spec["B"], spec["H"], 3)]
    for (l, b, h), (ro, rl) in oracle_frac_slices(inp, alphas, spec["base"], spec["W"], picks).items():
        assert max_abs(f64(o[l, b, h]), ro) <= TOL["bf16"], (l, b, h)
        assert max_abs(f64(lse[l, b, h]), rl) <= LSE_TOL["bf16"], (l, b, h)


FRAC_EDGE = [
    # (B, H, T, W, alpha, base)
    (1, 1, 1, 4, 1.37, "fib"),
    (1, 2, 2, 1, 0.61, "fib"),
    (2, 1, 63, 6, 1.37, "fib"),
    (1, 3, 127, 8, 0.77, "fib"),
    (1, 1, 129, 12, 2.3, "fib"),          # ragged last tile
    (2, 2, 1000, 10, 1.618, "fib"),
    (1, 2, 300, 64, 1.1, "pow2"),
    (1, 1, 700, 700, 1.3, "fib"),         # W >= T: no distance kept
    (1, 1, 1024, 1, 0.6, "fib"),          # distances sharing a ceiling
    (1, 2, 2049, 64, 3.7, "pow2"),
    (1, 1, 640, 16, 0.9999999, "fib"),    # weights just below 1
    (1, 1, 640, 16, 1.0000001, "fib"),    # weights just above 0
    (1, 1, 4096, 64, 0.8, "fib"),
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", FRAC_EDGE)
def test_fwd_frac_edge_cases(dtype, case):
    B, H, T, W, alpha, base = case
    inp = fi.draw((1, B, H, T, 64), seed=21 + T, scale=0.5, dtype=dtype)
    dev = to_dev(inp)
    o, lse = fa.fwd_frac(dev["q"], dev["k"], dev["v"], W, [alpha], base)
    torch.cuda.synchronize()
    fa.poll_device_error()
    picks = [(0, b, h) for b in range(B) for h in range(H)]
    for (l, b, h), (ro, rl) in oracle_frac_slices(inp, [alpha], base, W, picks).items():
        assert max_abs(f64(o[l, b, h]), ro) <= TOL[dtype]
        assert max_abs(f64(lse[l, b, h]), rl) <= LSE_TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("base", ["fib", "pow2"])
def test_fwd_frac_integer_alpha_equals_static_bitwise(dtype, base):
    inp = to_dev(fi.draw((3, 2, 2, 1000, 64), seed=31, scale=0.5, dtype=dtype))
    o, lse = fa.fwd_frac(inp["q"], inp["k"], inp["v"], 16, [1.0, 2.0, 3.0], base)
    for c, a in enumerate((1, 2, 3)):
        sc = fa.Schedule("fixed", base, alpha=(a, 1))
        os_, ls = fa.fwd(inp["q"][c], inp["k"][c], inp["v"][c], 16, sc)
        assert torch.equal(o[c], os_) and torch.equal(lse[c], ls), a


def test_fwd_frac_more_layers_than_one_launch_equals_per_layer_calls():
    n = 18
    alphas = [0.55 + 0.083 * l for l in range(n)]
    inp = to_dev(fi.draw((n, 1, 2, 300, 64), seed=41, scale=0.5, dtype="bf16"))
    o, lse = fa.fwd_frac(inp["q"], inp["k"], inp["v"], 8, alphas)
    for c in range(n):
        o1, l1 = fa.fwd_frac(inp["q"][c], inp["k"][c], inp["v"][c], 8, [alphas[c]])
        assert torch.equal(o1, o[c]) and torch.equal(l1, lse[c]), c


def test_fwd_frac_uniform_attention_over_linear_values():
    # Q = 0: every attended key weighs the same; V[j] = (a + b j) makes the interpolated
    # value at real position p equal a + b p, so O_i = a + b * mean(attended positions).
    T, W, alpha = 1000, 8, 1.37
    dists = oracle.frac_distances(f32(alpha), "fib", W, T)
    a = torch.linspace(-1, 1, 64, dtype=torch.float64)
    b = torch.linspace(0.5, -0.5, 64, dtype=torch.float64) / T
    v = (a[None, :] + torch.arange(T, dtype=torch.float64)[:, None] * b[None, :]).float()
    q = torch.zeros(1, 1, T, 64, device="cuda")
    k = torch.randn(1, 1, T, 64, device="cuda")
    o, lse = fa.fwd_frac(q, k, v.cuda()[None, None].contiguous(), W, [alpha])
    o = f64(o[0, 0])
    for i in range(T):
        pos = [float(j) for j in range(max(0, i - W + 1), i + 1)] + [i - d for d in dists if i >= d]
        want = (a + b * float(np.mean(pos))).numpy()
        assert np.abs(o[i] - want).max() <= TOL["f32"], i


def test_fwd_frac_deterministic():
    spec = fi.WORKLOADS["c3f"]
    inp = to_dev(fi.workload_inputs("c3f", layers=range(4), B=2))
    alphas = fi.frac_alphas(spec)[:4]
    a = fa.fwd_frac(inp["q"], inp["k"], inp["v"], 64, alphas)
    b = fa.fwd_frac(inp["q"], inp["k"], inp["v"], 64, alphas)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# ------------------------------------------------------------------ backward

DALPHA_TOL = {"f32": 1e-4, "bf16": 2e-2}  # relative to sum_t F_t |dL/dd_t| over the layer


def _frac_bwd_run(inp, W, alphas, base="fib"):
    dev = to_dev(inp)
    o, lse = fa.fwd_frac(dev["q"], dev["k"], dev["v"], W, alphas, base)
    dq, dk, dv, da = fa.bwd_frac(dev["q"], dev["k"], dev["v"], o, lse, dev["dO"], W, alphas, base)
    torch.cuda.synchronize()
    fa.poll_device_error()
    return o, dq, dk, dv, da


def _check_frac_bwd(inp, W, alphas, base, dtype, layers_full=None, picks=None):
    """Compare dq/dk/dv on picked slices and dalpha of fully recomputed layers."""
    o, dq, dk, dv, da = _frac_bwd_run(inp, W, alphas, base)
    Lc, B, H, T, _ = inp["q"].shape
    if picks is None:
        picks = [(l, b, h) for l in range(Lc) for b in range(B) for h in range(H)]
    if layers_full is None:
        layers_full = range(Lc)
    need = sorted(set(picks) | {(l, b, h) for l in layers_full for b in range(B) for h in range(H)})
    by_layer = {}
    for (l, b, h) in need:
        by_layer.setdefault(l, []).append((b, h))
    worst_o = 0.0
    for l, bhs in by_layer.items():
        a = f32(alphas[l])
        dists = oracle.frac_distances(a, base, W, T)
        fb = np.array(oracle.frac_bases(a, base, W, T), dtype=np.float64)
        g = lambda n: np.stack([f64(inp[n][l, b, h]) for b, h in bhs])
        rq, rk, rv, ro, rl, rdd = oracle.bwd_frac(g("q"), g("k"), g("v"), g("dO"), W, dists)
        for n, (b, h) in enumerate(bhs):
            if (l, b, h) in picks:
                assert_grad("dq", f64(dq[l, b, h]), rq[n], dtype, (l, b, h))
                assert_grad("dk", f64(dk[l, b, h]), rk[n], dtype, (l, b, h))
                assert_grad("dv", f64(dv[l, b, h]), rv[n], dtype, (l, b, h))
                worst_o = max(worst_o, max_abs(f64(o[l, b, h]), ro[n]))
        if l in layers_full and len(fb):
            ref = float((rdd[:, : len(fb)] * fb).sum())
            mag = float((np.abs(rdd[:, : len(fb)]) * fb).sum())
            err = abs(float(da[l]) - ref)
            assert err <= DALPHA_TOL[dtype] * max(mag, 1e-6), (l, float(da[l]), ref, mag)
    assert worst_o <= TOL[dtype], worst_o


FRAC_BWD_EDGE = [
    # (B, H, T, W, alpha, base)
    (1, 1, 1, 4, 1.37, "fib"),
    (1, 2, 2, 1, 0.61, "fib"),
    (2, 1, 63, 6, 1.37, "fib"),
    (1, 3, 127, 8, 0.77, "fib"),
    (1, 1, 129, 12, 2.3, "fib"),
    (2, 2, 1000, 10, 1.618, "fib"),
    (1, 2, 300, 64, 1.1, "pow2"),
    (1, 1, 700, 700, 1.3, "fib"),
    (1, 1, 1024, 1, 0.6, "fib"),
    (1, 2, 2049, 64, 3.7, "pow2"),
    (1, 1, 640, 16, 0.9999999, "fib"),
    (1, 1, 640, 16, 1.0000001, "fib"),
    (1, 1, 640, 16, 2.0, "fib"),          # integer alpha: the one-sided derivative
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", FRAC_BWD_EDGE)
def test_bwd_frac_edge_cases(dtype, case):
    B, H, T, W, alpha, base = case
    inp = fi.draw((1, B, H, T, 64), seed=61 + T, scale=0.5, dtype=dtype, names=("q", "k", "v", "dO"))
    _check_frac_bwd(inp, W, [alpha], base, dtype)


def test_bwd_frac_training_step_sampled():
    # the fractional workload's shape, forward + backward; dalpha of two layers in full
    spec = fi.WORKLOADS["c3f"]
    alphas = fi.frac_alphas(spec)
    inp = fi.workload_inputs("c3f", names=("q", "k", "v", "dO"))
    picks = [(l, b, h) for l in range(spec["Lc"]) for (b, h) in sample_slices(spec["B"], spec["H"], 2)]
    _check_frac_bwd(inp, spec["W"], alphas, spec["base"], "bf16", layers_full=[0, 15], picks=picks)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_bwd_frac_integer_alpha_equals_static_bitwise(dtype):
    inp = to_dev(fi.draw((2, 2, 2, 700, 64), seed=71, scale=0.5, dtype=dtype,
                         names=("q", "k", "v", "dO")))
    o, lse = fa.fwd_frac(inp["q"], inp["k"], inp["v"], 16, [1.0, 3.0])
    dq, dk, dv, _ = fa.bwd_frac(inp["q"], inp["k"], inp["v"], o, lse, inp["dO"], 16, [1.0, 3.0])
    for c, a in enumerate((1, 3)):
        sc = fa.Schedule("fixed", "fib", alpha=(a, 1))
        g = fa.bwd(inp["q"][c], inp["k"][c], inp["v"][c], o[c], lse[c], inp["dO"][c], 16, sc)
        assert torch.equal(dq[c], g[0]) and torch.equal(dk[c], g[1]) and torch.equal(dv[c], g[2]), a


def test_bwd_frac_more_layers_than_one_launch_equals_per_layer_calls():
    n = 18
    alphas = [0.55 + 0.083 * l for l in range(n)]
    inp = to_dev(fi.draw((n, 1, 2, 300, 64), seed=81, scale=0.5, dtype="bf16",
                         names=("q", "k", "v", "dO")))
    o, lse = fa.fwd_frac(inp["q"], inp["k"], inp["v"], 8, alphas)
    dq, dk, dv, da = fa.bwd_frac(inp["q"], inp["k"], inp["v"], o, lse, inp["dO"], 8, alphas)
    for c in range(n):
        g = fa.bwd_frac(inp["q"][c], inp["k"][c], inp["v"][c], o[c], lse[c], inp["dO"][c], 8,
                        [alphas[c]])
        assert torch.equal(dq[c], g[0]) and torch.equal(dk[c], g[1]) and torch.equal(dv[c], g[2])
        assert torch.equal(da[c:c + 1], g[3]), c


def test_bwd_frac_deterministic():
    spec = fi.WORKLOADS["c3f"]
    inp = to_dev(fi.workload_inputs("c3f", layers=range(3), B=2, names=("q", "k", "v", "dO")))
    alphas = fi.frac_alphas(spec)[:3]
    o, lse = fa.fwd_frac(inp["q"], inp["k"], inp["v"], 64, alphas)
    a = fa.bwd_frac(inp["q"], inp["k"], inp["v"], o, lse, inp["dO"], 64, alphas)
    b = fa.bwd_frac(inp["q"], inp["k"], inp["v"], o, lse, inp["dO"], 64, alphas)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_frac_autograd_wrapper_gives_alpha_gradient():
    inp = to_dev(fi.draw((2, 1, 2, 400, 64), seed=91, scale=0.5, dtype="bf16",
                         names=("q", "k", "v", "dO")))
    alpha = torch.tensor([0.9, 1.45], dtype=torch.float32, requires_grad=True)
    q, k, v = (inp[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
    o = fa.FibFracAttention.apply(q, k, v, alpha, 16)
    o.backward(inp["dO"])
    o2, lse = fa.fwd_frac(inp["q"], inp["k"], inp["v"], 16, [0.9, 1.45])
    dq, dk, dv, da = fa.bwd_frac(inp["q"], inp["k"], inp["v"], o2, lse, inp["dO"], 16, [0.9, 1.45])
    assert torch.equal(o.detach(), o2)
    assert torch.equal(q.grad, dq) and torch.equal(k.grad, dk) and torch.equal(v.grad, dv)
    assert torch.equal(alpha.grad, da.cpu())
