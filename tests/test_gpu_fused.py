"""GPU parity of the one-pass backward (fibattn_bwd_fused): one thread block per 128-row tile
writes dq of its queries and dk, dv of its keys, forming each diagonal pair again on the key
side. Checked against the fp64 oracle under the absolute and the relative gate, and against
the two-kernel backward (fibattn_bwd) bit for bit, which forms every P and dS from the same
operands in the same order and sums in the same order (needs a B300)."""
import pytest
import torch

import fibattn_inputs as fi
import static_fibonacci_offset_fibattn_b300 as fa
from gpu_common import (assert_grad, f64, lib_schedule, oracle_bwd_slices, oracle_table,
                        sample_slices, to_dev)
from test_gpu_parity import BWD_EDGE, SCHEDS

pytestmark = pytest.mark.gpu


def _both(dev, W, sc, layer0=0, workspace=None):
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], W, sc, layer0=layer0)
    g_fused = fa.bwd_fused(dev["q"], dev["k"], dev["v"], o, lse, dev["dO"], W, sc, layer0=layer0,
                           workspace=workspace)
    g_split = fa.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["dO"], W, sc, layer0=layer0)
    torch.cuda.synchronize()
    fa.poll_device_error()
    return g_fused, g_split


def _assert_equal(g_fused, g_split):
    for n, a, b in zip(("dq", "dk", "dv"), g_fused, g_split):
        if not torch.equal(a, b):
            diff = (a.float() - b.float()).abs()
            raise AssertionError(f"{n}: fused and two-kernel backward differ at "
                                 f"{int((diff > 0).sum())} elements, max {float(diff.max()):.3g}")


def _run_workload(name, picks_per_layer, **override):
    spec = dict(fi.WORKLOADS[name], **override)
    inp = fi.workload_inputs(name, **override)
    dev = to_dev(inp)
    sc = lib_schedule(spec["sched"])
    g_fused, g_split = _both(dev, spec["W"], sc)
    picks = [(l, b, h) for l in range(spec["Lc"])
             for (b, h) in sample_slices(spec["B"], spec["H"], picks_per_layer)]
    ref = oracle_bwd_slices(inp, spec["sched"], spec["W"], 0, picks)
    worst = {n: (0.0, 0.0) for n in ("dq", "dk", "dv")}
    for (l, b, h), (rq, rk, rv, ro, rl) in ref.items():
        for n, got, want in zip(("dq", "dk", "dv"), g_fused, (rq, rk, rv)):
            err, rel = assert_grad(n, f64(got[l, b, h]), want, "bf16", (l, b, h))
            worst[n] = (max(worst[n][0], err), max(worst[n][1], rel))
    print(f"fused {name} {override or ''} backward worst (max-abs, relative):",
          {n: (float(f"{e:.3g}"), float(f"{r:.3g}")) for n, (e, r) in worst.items()})
    return g_fused, g_split


def test_fused_bwd_c5_training_step_sampled():
    g_fused, g_split = _run_workload("c5", 2)
    _assert_equal(g_fused, g_split)


def test_fused_bwd_c5_large_gradients_sampled():
    # inputs four times larger (N(0,1)/2): gradients far from the absolute bound's floor
    g_fused, g_split = _run_workload("c5", 2, scale=0.5)
    _assert_equal(g_fused, g_split)


def test_fused_bwd_c5_pow2_and_linear_schedules():
    # every layer of the power-of-two control and of the linear stagger, against the split
    for sched in (SCHEDS[1], SCHEDS[2]):
        inp = to_dev(fi.draw((16, 1, 2, 1024, 64), seed=41, scale=0.5, dtype="bf16",
                             names=("q", "k", "v", "dO")))
        _assert_equal(*_both(inp, 64, lib_schedule(sched)))


@pytest.mark.parametrize("case", BWD_EDGE)
def test_fused_bwd_edge_cases(case):
    # one row, ragged tails, W >= T (dense), W > 64 (band chunks through the ring on both
    # sides), W = 1, a last tile of one row, an uncapped Fibonacci base
    B, H, T, W, sched = case
    layer = sched["n_layers"] - 1
    inp = fi.draw((1, B, H, T, 64), seed=21 + T, scale=0.25, dtype="bf16",
                  names=("q", "k", "v", "dO"))
    dev = to_dev(inp)
    g_fused, g_split = _both(dev, W, lib_schedule(sched), layer0=layer)
    picks = [(0, b, h) for b in range(B) for h in range(H)]
    ref = oracle_bwd_slices(inp, sched, W, layer, picks)
    for (l, b, h), (rq, rk, rv, ro, rl) in ref.items():
        for n, got, want in zip(("dq", "dk", "dv"), g_fused, (rq, rk, rv)):
            assert_grad(n, f64(got[l, b, h]), want, "bf16", (b, h))
    _assert_equal(g_fused, g_split)


@pytest.mark.parametrize("TW", [(1000, 200), (700, 129), (2048, 700), (300, 1)])
def test_fused_bwd_wide_windows(TW):
    # windows wider than a tile: several band chunks below (dq) and past (dk/dv) the tile
    T, W = TW
    sched = SCHEDS[4]
    inp = fi.draw((1, 1, 2, T, 64), seed=61 + W, scale=0.5, dtype="bf16",
                  names=("q", "k", "v", "dO"))
    dev = to_dev(inp)
    g_fused, g_split = _both(dev, W, lib_schedule(sched), layer0=3)
    ref = oracle_bwd_slices(inp, sched, W, 3, [(0, 0, h) for h in range(2)])
    for (l, b, h), (rq, rk, rv, ro, rl) in ref.items():
        for n, got, want in zip(("dq", "dk", "dv"), g_fused, (rq, rk, rv)):
            assert_grad(n, f64(got[l, b, h]), want, "bf16", h)
    _assert_equal(g_fused, g_split)


def test_fused_bwd_empty_table_is_sliding_window_gradient():
    sched = dict(kind="fixed", base="fib", alpha=(1, 1), n_layers=1, base_max=10)
    assert oracle_table(sched, 0, 16, 500) == []
    inp = fi.draw((1, 1, 2, 500, 64), seed=23, scale=0.25, dtype="bf16", names=("q", "k", "v", "dO"))
    dev = to_dev(inp)
    g_fused, g_split = _both(dev, 16, lib_schedule(sched))
    ref = oracle_bwd_slices(inp, sched, 16, 0, [(0, 0, h) for h in range(2)])
    for (l, b, h), (rq, rk, rv, ro, rl) in ref.items():
        for n, got, want in zip(("dq", "dk", "dv"), g_fused, (rq, rk, rv)):
            assert_grad(n, f64(got[l, b, h]), want, "bf16", h)
    _assert_equal(g_fused, g_split)


def test_fused_bwd_more_layers_than_one_launch():
    # 18 layers: launches of 16 + 2 layers, each with its own workspace rows
    sched = dict(kind="linear", base="fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=20)
    inp = to_dev(fi.draw((18, 1, 2, 400, 64), seed=25, scale=0.25, dtype="bf16",
                         names=("q", "k", "v", "dO")))
    _assert_equal(*_both(inp, 64, lib_schedule(sched), layer0=1))


def test_fused_bwd_workspace_contents_do_not_matter():
    # a NaN-filled workspace (and the fused call's smallest workspace size) gives the same
    # bits: the pre-pass writes every D and lse row, pad rows included
    inp = to_dev(fi.draw((2, 1, 2, 777, 64), seed=27, scale=0.5, dtype="bf16",
                         names=("q", "k", "v", "dO")))
    sc = lib_schedule(SCHEDS[4])
    ws = torch.full((fa.bwd_fused_workspace_size(inp["q"]) // 4,), float("nan"), device="cuda")
    g_nan, g_split = _both(inp, 64, sc, workspace=ws.view(torch.uint8))
    _assert_equal(g_nan, g_split)


def test_fused_bwd_deterministic_and_on_a_side_stream():
    inp = to_dev(fi.workload_inputs("c5", layers=range(2), B=2))
    sc = lib_schedule(fi.WORKLOADS["c5"]["sched"])
    o, lse = fa.fwd(inp["q"], inp["k"], inp["v"], 64, sc)
    a = fa.bwd_fused(inp["q"], inp["k"], inp["v"], o, lse, inp["dO"], 64, sc)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        b = fa.bwd_fused(inp["q"], inp["k"], inp["v"], o, lse, inp["dO"], 64, sc)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    _assert_equal(a, b)


def test_fused_bwd_rejects_unsupported_shapes():
    q = torch.zeros(1, 1, 1, 64, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FibAttnError):
        fa.bwd_fused(q, q, q, q, torch.zeros(1, 1, 1, 64, device="cuda"), q, 16, fa.Schedule())
    q32 = torch.zeros(1, 1, 1, 64, 64, device="cuda")
    with pytest.raises(fa.FibAttnError):
        fa.bwd_fused(q32, q32, q32, q32, torch.zeros(1, 1, 1, 64, device="cuda"), q32, 16,
                     fa.Schedule())
