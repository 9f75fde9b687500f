"""GPU parity: the CUDA path through the C ABI against the oracle (needs a B300).

Index work is compared bit-exactly (offset tables, key sets); values within the
stated max-abs tolerances (1e-5 fp32 path, 2e-2 bf16 path). Full-size workloads run
in the same launch configuration the benchmark times, and sampled slices are
recomputed by the oracle.
"""
import math

import numpy as np
import pytest
import torch

import fibattn_inputs as fi
import oracle
import static_fibonacci_offset_fibattn_b300 as fa
from gpu_common import (LSE_TOL, TOL, assert_grad, f64, lib_schedule, max_abs,
                        oracle_bwd_slices, oracle_fwd_slices, oracle_table, sample_slices,
                        to_dev)

pytestmark = pytest.mark.gpu

SCHEDS = [
    dict(kind="fixed", base="fib", alpha=(1, 1), n_layers=1),
    dict(kind="fixed", base="pow2", alpha=(1, 1), n_layers=16),
    dict(kind="linear", base="fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=16),
    dict(kind="linear", base="fib", alpha_min=(1, 2), alpha_max=(3, 2), n_layers=16),
    dict(kind="coprime", base="fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=16, coprime_c=5),
    dict(kind="coprime", base="fib", alpha_min=(1, 2), alpha_max=(3, 2), n_layers=16, coprime_c=7),
    dict(kind="linear", base="pow2", alpha_min=(1, 2), alpha_max=(3, 2), n_layers=16),
    dict(kind="fixed", base="fib", alpha=(7, 3), n_layers=1, base_max=100000),
    dict(kind="coprime", base="pow2", alpha_min=(1, 7), alpha_max=(9, 4), n_layers=9, coprime_c=4),
]


@pytest.mark.parametrize("sched", SCHEDS)
@pytest.mark.parametrize("WT", [(16, 256), (64, 1024), (64, 4096), (6, 1024), (12, 100000)])
def test_device_tables_bit_exact(sched, WT):
    W, T = WT
    L = sched["n_layers"]
    tab, cnt = fa.offsets_device(lib_schedule(sched), 0, L, W, T)
    tab, cnt = tab.cpu().tolist(), cnt.cpu().tolist()
    for l in range(L):
        want = oracle_table(sched, l, W, T)
        assert cnt[l] == len(want)
        assert tab[l][: cnt[l]] == want
        assert all(x == -1 for x in tab[l][cnt[l]:])
        assert fa.offsets(lib_schedule(sched), l, W, T) == want


@pytest.mark.parametrize("WT", [(16, 256), (6, 300), (64, 1024), (1, 100), (300, 257)])
@pytest.mark.parametrize("sched", SCHEDS[:5])
def test_keyset_debug_matches_oracle(sched, WT):
    W, T = WT
    for l in sorted({0, sched["n_layers"] - 1}):
        m = fa.keyset_debug(lib_schedule(sched), l, W, T).cpu().numpy()
        tab = oracle_table(sched, l, W, T)
        for i in range(T):
            assert np.flatnonzero(m[i]).tolist() == oracle.key_set(i, W, tab), (l, i)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("WT", [(16, 256), (64, 640), (6, 300)])
def test_keyset_probe_through_forward(dtype, WT):
    # Black box: Q = 0 makes every attended key weigh 1/|S_i|; V = one-hot over a block of
    # 64 keys makes |S_i| * O_i[c] = [key 64*blk + c in S_i]. LSE_i = ln |S_i|.
    W, T = WT
    sched = dict(kind="linear", base="fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=16)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    layer = 9
    tab = oracle_table(sched, layer, W, T)
    want = np.zeros((T, T), dtype=bool)
    for i in range(T):
        want[i, oracle.key_set(i, W, tab)] = True
    got = np.zeros((T, T), dtype=bool)
    q = torch.zeros(1, 1, T, 64, dtype=dt, device="cuda")
    k = torch.randn(1, 1, T, 64, device="cuda").to(dt)
    for blk in range((T + 63) // 64):
        v = torch.zeros(1, 1, T, 64, dtype=dt, device="cuda")
        for c in range(64):
            j = 64 * blk + c
            if j < T:
                v[0, 0, j, c] = 1
        o, lse = fa.fwd(q, k, v, W, lib_schedule(sched), layer0=layer)
        n = torch.exp(lse[0, 0].double())
        cnt = want.sum(1)
        assert np.max(np.abs(n.cpu().numpy() - cnt)) < 1e-3 * cnt.max()
        frac = (o[0, 0].double() * torch.from_numpy(cnt).cuda()[:, None]).cpu().numpy()
        hi = min(T, 64 * blk + 64)
        got[:, 64 * blk: hi] = frac[:, : hi - 64 * blk] > 0.5
    assert (got == want).all()


def _run_fwd(name, picks_per_layer, **override):
    spec = dict(fi.WORKLOADS[name], **override)
    inp = fi.workload_inputs(name, **override)
    dev = to_dev(inp)
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], spec["W"], lib_schedule(spec["sched"]))
    torch.cuda.synchronize()
    fa.poll_device_error()
    picks = [(l, b, h) for l in range(spec["Lc"])
             for (b, h) in sample_slices(spec["B"], spec["H"], picks_per_layer)]
    ref = oracle_fwd_slices(inp, spec["sched"], spec["W"], 0, picks)
    worst_o = worst_l = 0.0
    for (l, b, h), (ro, rl) in ref.items():
        worst_o = max(worst_o, max_abs(f64(o[l, b, h]), ro))
        worst_l = max(worst_l, max_abs(f64(lse[l, b, h]), rl))
    return spec, worst_o, worst_l


def test_fwd_c1_fp32_all_slices():
    spec, eo, el = _run_fwd("c1", 64)
    assert eo <= TOL["f32"], eo
    assert el <= LSE_TOL["f32"], el


def test_fwd_c2_bf16_all_slices():
    spec, eo, el = _run_fwd("c2", 64)
    assert eo <= TOL["bf16"], eo
    assert el <= LSE_TOL["bf16"], el


@pytest.mark.parametrize("name", ["c3", "c3p"])
def test_fwd_c3_sixteen_layers_sampled(name):
    spec, eo, el = _run_fwd(name, 3)
    assert eo <= TOL["bf16"], eo
    assert el <= LSE_TOL["bf16"], el


def test_fwd_c4_extrapolation_sampled():
    spec, eo, el = _run_fwd("c4", 2)
    assert eo <= TOL["bf16"], eo
    assert el <= LSE_TOL["bf16"], el


EDGE = [
    # (B, H, T, W, sched)
    (1, 1, 1, 4, SCHEDS[0]),
    (1, 2, 2, 1, SCHEDS[0]),
    (2, 1, 63, 6, SCHEDS[2]),
    (1, 3, 127, 8, SCHEDS[3]),
    (1, 1, 129, 12, SCHEDS[4]),
    (2, 2, 1000, 10, SCHEDS[5]),
    (1, 2, 300, 64, SCHEDS[1]),
    (1, 1, 700, 700, SCHEDS[0]),       # W >= T: dense causal
    (1, 1, 333, 5000, SCHEDS[2]),      # W > T
    (2, 1, 515, 100, SCHEDS[2]),       # W > 64
    (1, 1, 1024, 1, SCHEDS[0]),        # window = the query itself
    (1, 2, 2049, 64, SCHEDS[6]),
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", EDGE)
def test_fwd_edge_cases(dtype, case):
    B, H, T, W, sched = case
    layer = sched["n_layers"] - 1
    sched_one = dict(sched)
    inp = fi.draw((1, B, H, T, 64), seed=11 + T, scale=0.5, dtype=dtype)
    dev = to_dev(inp)
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], W, lib_schedule(sched_one), layer0=layer)
    torch.cuda.synchronize()
    picks = [(0, b, h) for b in range(B) for h in range(H)]
    ref = oracle_fwd_slices(inp, sched_one, W, layer, picks)
    for (l, b, h), (ro, rl) in ref.items():
        assert max_abs(f64(o[l, b, h]), ro) <= TOL[dtype]
        assert max_abs(f64(lse[l, b, h]), rl) <= LSE_TOL[dtype]


def test_fwd_empty_table_is_sliding_window():
    sched = dict(kind="fixed", base="fib", alpha=(1, 1), n_layers=1, base_max=10)
    inp = fi.draw((1, 2, 2, 500, 64), seed=5, scale=0.5, dtype="bf16")
    assert oracle_table(sched, 0, 16, 500) == []
    dev = to_dev(inp)
    o, _ = fa.fwd(dev["q"], dev["k"], dev["v"], 16, lib_schedule(sched))
    T = 500
    band = torch.ones(T, T, dtype=torch.bool).tril() & ~torch.ones(T, T, dtype=torch.bool).tril(-16)
    ref = torch.nn.functional.scaled_dot_product_attention(
        inp["q"].double(), inp["k"].double(), inp["v"].double(), attn_mask=band)
    assert max_abs(f64(o), ref.numpy()) <= TOL["bf16"]


def test_fwd_dense_causal_matches_sdpa():
    inp = fi.draw((1, 2, 4, 1024, 64), seed=6, scale=0.125, dtype="bf16")
    dev = to_dev(inp)
    o, _ = fa.fwd(dev["q"], dev["k"], dev["v"], 1024, lib_schedule(SCHEDS[0]))
    ref = torch.nn.functional.scaled_dot_product_attention(
        dev["q"][0], dev["k"][0], dev["v"][0], is_causal=True)
    assert max_abs(f64(o[0]), f64(ref)) <= TOL["bf16"]


def test_fwd_dense_causal_at_4x_length():
    # the dense causal context at the 4x-length shape (one layer of those inputs, W = T = 4096):
    # no offset survives, so the forward is dense causal attention; against torch's SDPA on the
    # same tensors and, on two slices, the oracle
    spec = fi.WORKLOADS["c4"]
    inp = fi.workload_inputs("c4", layers=[0])
    dev = to_dev(inp)
    T = spec["T"]
    sc = lib_schedule(spec["sched"])
    assert fa.offsets(sc, 0, T, T) == []
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], T, sc)
    torch.cuda.synchronize()
    fa.poll_device_error()
    ref = torch.nn.functional.scaled_dot_product_attention(
        dev["q"][0].float(), dev["k"][0].float(), dev["v"][0].float(), is_causal=True)
    assert max_abs(f64(o[0]), f64(ref)) <= TOL["bf16"]
    picks = [(0, 0, 0), (0, 1, 7)]
    for (l, b, h), (ro, rl) in oracle_fwd_slices(inp, spec["sched"], T, 0, picks).items():
        assert max_abs(f64(o[l, b, h]), ro) <= TOL["bf16"]
        assert max_abs(f64(lse[l, b, h]), rl) <= LSE_TOL["bf16"]


def test_fwd_layer_batched_equals_per_layer_calls():
    spec = fi.WORKLOADS["c3"]
    inp = to_dev(fi.workload_inputs("c3", layers=range(4), B=2, H=2))
    sc = lib_schedule(spec["sched"])
    o_all, l_all = fa.fwd(inp["q"], inp["k"], inp["v"], 64, sc, layer0=3)
    for c in range(4):
        o1, l1 = fa.fwd(inp["q"][c], inp["k"][c], inp["v"][c], 64, sc, layer0=3 + c)
        assert torch.equal(o1, o_all[c]) and torch.equal(l1, l_all[c])


def test_fwd_on_side_stream():
    inp = to_dev(fi.draw((1, 1, 2, 777, 64), seed=9, scale=0.125, dtype="bf16"))
    o0, _ = fa.fwd(inp["q"], inp["k"], inp["v"], 64, lib_schedule(SCHEDS[0]))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1, _ = fa.fwd(inp["q"], inp["k"], inp["v"], 64, lib_schedule(SCHEDS[0]))
    s.synchronize()
    assert torch.equal(o0, o1)


def test_fwd_deterministic():
    inp = to_dev(fi.workload_inputs("c2", B=2))
    sc = lib_schedule(fi.WORKLOADS["c2"]["sched"])
    a = fa.fwd(inp["q"], inp["k"], inp["v"], 64, sc)
    b = fa.fwd(inp["q"], inp["k"], inp["v"], 64, sc)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# ------------------------------------------------------------------ backward

def _run_bwd(name, picks_per_layer, **override):
    """Forward and backward of a whole workload in the bench's launch configuration; every
    picked slice's dq, dk, dv against the oracle under the absolute and the relative gate.
    Returns the worst max-abs error and relative error per tensor (printed, for the record)."""
    spec = dict(fi.WORKLOADS[name], **override)
    inp = fi.workload_inputs(name, **override)
    dev = to_dev(inp)
    sc = lib_schedule(spec["sched"])
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], spec["W"], sc)
    dq, dk, dv = fa.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["dO"], spec["W"], sc)
    torch.cuda.synchronize()
    fa.poll_device_error()
    picks = [(l, b, h) for l in range(spec["Lc"])
             for (b, h) in sample_slices(spec["B"], spec["H"], picks_per_layer)]
    ref = oracle_bwd_slices(inp, spec["sched"], spec["W"], 0, picks)
    worst = {n: (0.0, 0.0) for n in ("dq", "dk", "dv")}
    worst_o = 0.0
    for (l, b, h), (rq, rk, rv, ro, rl) in ref.items():
        for n, got, want in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
            err, rel = assert_grad(n, f64(got[l, b, h]), want, "bf16", (l, b, h))
            worst[n] = (max(worst[n][0], err), max(worst[n][1], rel))
        worst_o = max(worst_o, max_abs(f64(o[l, b, h]), ro))
    assert worst_o <= TOL["bf16"], worst_o
    print(f"{name} {override or ''} backward worst (max-abs, relative):",
          {n: (float(f"{e:.3g}"), float(f"{r:.3g}")) for n, (e, r) in worst.items()})
    return worst


def test_bwd_c5_training_step_sampled():
    _run_bwd("c5", 2)


def test_bwd_c5_training_step_large_gradients_sampled():
    # the same full-size step (every persistent CTA takes many tiles) with inputs four times
    # larger (N(0,1)/2), where the gradients are far from the absolute bound's floor
    _run_bwd("c5", 2, scale=0.5)


BWD_EDGE = [
    (1, 1, 1, 4, SCHEDS[0]),
    (1, 2, 63, 6, SCHEDS[2]),
    (2, 1, 129, 12, SCHEDS[4]),
    (1, 1, 1000, 64, SCHEDS[5]),
    (1, 1, 300, 300, SCHEDS[0]),       # W >= T: dense causal
    (1, 2, 517, 100, SCHEDS[1]),       # W > 64
    (1, 1, 1024, 1, SCHEDS[0]),        # window = the query itself
    (1, 1, 2049, 64, SCHEDS[6]),       # last tile holds one row
    (1, 1, 640, 16, SCHEDS[7]),        # alpha 7/3 over an uncapped Fibonacci base
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", BWD_EDGE)
def test_bwd_edge_cases(dtype, case):
    B, H, T, W, sched = case
    layer = sched["n_layers"] - 1
    inp = fi.draw((1, B, H, T, 64), seed=21 + T, scale=0.25, dtype=dtype,
                  names=("q", "k", "v", "dO"))
    dev = to_dev(inp)
    sc = lib_schedule(sched)
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], W, sc, layer0=layer)
    dq, dk, dv = fa.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["dO"], W, sc, layer0=layer)
    torch.cuda.synchronize()
    picks = [(0, b, h) for b in range(B) for h in range(H)]
    ref = oracle_bwd_slices(inp, sched, W, layer, picks)
    for (l, b, h), (rq, rk, rv, ro, rl) in ref.items():
        for n, got, want in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
            assert_grad(n, f64(got[l, b, h]), want, dtype, (b, h))


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("f32", 64), ("bf16", 128)])
def test_window_at_the_int32_limit_equals_a_window_of_T(dtype, d):
    # a window of T keys already holds every causal key, so W = 2^31 - 1 must give the same
    # forward and backward, bit for bit (the window is clamped to T before the kernels' 32-bit
    # row arithmetic sees it)
    T = 300
    inp = to_dev(fi.draw((1, 1, 2, T, d), seed=41, scale=0.5, dtype=dtype,
                         names=("q", "k", "v", "dO")))
    sc = lib_schedule(SCHEDS[2])
    outs = []
    for W in (T, 2 ** 31 - 1):
        o, lse = fa.fwd(inp["q"], inp["k"], inp["v"], W, sc, layer0=15)
        grads = fa.bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["dO"], W, sc, layer0=15)
        outs.append((o, lse) + tuple(grads))
    torch.cuda.synchronize()
    fa.poll_device_error()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_autograd_wrapper_matches_bwd():
    inp = to_dev(fi.draw((1, 2, 1, 300, 64), seed=31, scale=0.25, dtype="bf16",
                         names=("q", "k", "v", "dO")))
    sc = lib_schedule(SCHEDS[2])
    q, k, v = (inp[n][0].clone().requires_grad_() for n in "qkv")
    o = fa.FibSparseAttention.apply(q, k, v, 64, sc, 4)
    o.backward(inp["dO"][0])
    o2, lse = fa.fwd(inp["q"][0], inp["k"][0], inp["v"][0], 64, sc, layer0=4)
    dq, dk, dv = fa.bwd(inp["q"][0], inp["k"][0], inp["v"][0], o2, lse, inp["dO"][0], 64, sc, 4)
    assert torch.equal(o, o2) and torch.equal(q.grad, dq) and torch.equal(k.grad, dk)
    assert torch.equal(v.grad, dv)


def test_bwd_empty_table_is_sliding_window_gradient():
    # no offsets at all (base_max < W): the backward of plain sliding-window attention
    sched = dict(kind="fixed", base="fib", alpha=(1, 1), n_layers=1, base_max=10)
    assert oracle_table(sched, 0, 16, 500) == []
    inp = fi.draw((1, 1, 2, 500, 64), seed=23, scale=0.25, dtype="bf16", names=("q", "k", "v", "dO"))
    dev = to_dev(inp)
    sc = lib_schedule(sched)
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], 16, sc)
    dq, dk, dv = fa.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["dO"], 16, sc)
    ref = oracle_bwd_slices(inp, sched, 16, 0, [(0, 0, h) for h in range(2)])
    for (l, b, h), (rq, rk, rv, ro, rl) in ref.items():
        for n, got, want in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
            assert_grad(n, f64(got[l, b, h]), want, "bf16", h)


def test_bwd_more_layers_than_one_launch_equals_per_layer_calls():
    # 18 layers: the call is split into launches of 16 + 2 layers sharing one workspace
    sched = dict(kind="linear", base="fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=20)
    sc = lib_schedule(sched)
    inp = to_dev(fi.draw((18, 1, 2, 400, 64), seed=25, scale=0.25, dtype="bf16",
                         names=("q", "k", "v", "dO")))
    o, lse = fa.fwd(inp["q"], inp["k"], inp["v"], 64, sc, layer0=1)
    dq, dk, dv = fa.bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["dO"], 64, sc, layer0=1)
    for c in (0, 15, 16, 17):
        g = fa.bwd(inp["q"][c], inp["k"][c], inp["v"][c], o[c], lse[c], inp["dO"][c], 64, sc,
                   layer0=1 + c)
        assert torch.equal(g[0], dq[c]) and torch.equal(g[1], dk[c]) and torch.equal(g[2], dv[c])


def test_bwd_deterministic():
    inp = to_dev(fi.workload_inputs("c5", layers=range(2), B=2))
    sc = lib_schedule(fi.WORKLOADS["c5"]["sched"])
    o, lse = fa.fwd(inp["q"], inp["k"], inp["v"], 64, sc)
    a = fa.bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["dO"], 64, sc)
    b = fa.bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["dO"], 64, sc)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_fwd_bwd_from_a_fresh_host_thread():
    # a host thread that has made no CUDA runtime call yet has no current context; the
    # launchers must bind it before encoding their TMA tensor maps
    import threading

    inp = to_dev(fi.draw((1, 1, 2, 300, 64), seed=33, scale=0.25, dtype="bf16",
                         names=("q", "k", "v", "dO")))
    sc = lib_schedule(SCHEDS[2])
    o0, l0 = fa.fwd(inp["q"], inp["k"], inp["v"], 64, sc, layer0=4)
    g0 = fa.bwd(inp["q"], inp["k"], inp["v"], o0, l0, inp["dO"], 64, sc, layer0=4)
    torch.cuda.synchronize()
    out = {}

    def work():
        try:
            o, l = fa.fwd(inp["q"], inp["k"], inp["v"], 64, sc, layer0=4)
            g = fa.bwd(inp["q"], inp["k"], inp["v"], o, l, inp["dO"], 64, sc, layer0=4)
            torch.cuda.synchronize()
            out["res"] = (o, l, *g)
        except Exception as e:  # reported on the main thread
            out["err"] = e

    t = threading.Thread(target=work)
    t.start()
    t.join()
    assert "err" not in out, out.get("err")
    for a, b in zip(out["res"], (o0, l0, *g0)):
        assert torch.equal(a, b)
