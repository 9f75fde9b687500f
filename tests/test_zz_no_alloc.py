"""fibattn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: an operator hosted by a framework that owns the
device allocator and passes it no workspace, or a latency-critical loop where
cudaMalloc/cudaFree would synchronise the device. fibattn_bwd needs a caller-allocated
workspace (D per row and the (P, dS) pair of every diagonal entry); fibattn_bwd_noalloc
takes it from a fixed 40 MiB per-device array inside the library instead. Both run the
same deterministic kernels, so these tests call it through the C ABI and require its
results to equal fibattn_bwd's bit for bit: on two calls in a row (the array keeps the
previous call's contents), on the fp32 path, and after a call that left non-finite
values where the next call reads bytes it does not write (the pad rows past T).

This file is collected last on purpose, so that a run stopping at its first failure has
already run every other test.
"""
import pytest
import torch

import fibattn_inputs as fi
import static_fibonacci_offset_fibattn_b300 as fa

pytestmark = pytest.mark.gpu

SCHED = fa.Schedule("coprime", "fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=16, coprime_c=5)


def _inputs(shape, seed, dtype="bf16"):
    inp = fi.draw(shape, seed=seed, scale=0.125, dtype=dtype, names=("q", "k", "v", "dO"))
    return {n: t.cuda() for n, t in inp.items()}


def _assert_same(want, got):
    torch.cuda.synchronize()
    fa.poll_device_error()
    for name, a, b in zip(("dq", "dk", "dv"), want, got):
        assert torch.equal(a, b), (name, float((a.float() - b.float()).abs().max()))


def _compare(x, layer0=0):
    o, lse = fa.fwd(x["q"], x["k"], x["v"], 64, SCHED, layer0=layer0)
    want = fa.bwd(x["q"], x["k"], x["v"], o, lse, x["dO"], 64, SCHED, layer0=layer0)
    got = fa.bwd_noalloc(x["q"], x["k"], x["v"], o, lse, x["dO"], 64, SCHED, layer0=layer0)
    _assert_same(want, got)


def test_noalloc_matches_bwd_on_two_calls_in_a_row():
    # two different inputs back to back: the second call must not see the first's workspace
    _compare(_inputs((2, 2, 4, 1024, 64), seed=41), layer0=3)
    _compare(_inputs((3, 1, 2, 777, 64), seed=42), layer0=9)


def test_noalloc_matches_bwd_on_the_fp32_path():
    _compare(_inputs((2, 1, 2, 300, 64), seed=45, dtype="f32"), layer0=4)
    _compare(_inputs((1, 2, 1, 129, 64), seed=46, dtype="f32"), layer0=11)


def test_noalloc_after_a_call_that_left_non_finite_values():
    # A first call with NaN upstream gradients and NaN lse writes NaN into every workspace
    # value it produces: D, lse * log2(e) and the (P, dS) pairs, over the first 64 KB of the
    # array and more. The next call (T = 777, rows padded to 780) reads the pad rows 777-779
    # of D and lse * log2(e) without writing them, and pairs of queries past T: all of it
    # lies in that poisoned range. Its results must equal fibattn_bwd's with a zeroed
    # workspace, and fibattn_bwd's with a NaN-filled one.
    p = _inputs((1, 1, 8, 1024, 64), seed=47)
    o, lse = fa.fwd(p["q"], p["k"], p["v"], 64, SCHED)
    nan_dO = torch.full_like(p["dO"], float("nan"))
    nan_lse = torch.full_like(lse, float("nan"))
    fa.bwd_noalloc(p["q"], p["k"], p["v"], o, nan_lse, nan_dO, 64, SCHED)
    torch.cuda.synchronize()
    fa.poll_device_error()

    x = _inputs((1, 1, 2, 777, 64), seed=48)
    o, lse = fa.fwd(x["q"], x["k"], x["v"], 64, SCHED, layer0=15)
    got = fa.bwd_noalloc(x["q"], x["k"], x["v"], o, lse, x["dO"], 64, SCHED, layer0=15)
    need = fa.bwd_workspace_size(x["q"], 64, SCHED, 15)
    assert need <= 64 << 10
    for fill in (0, 0xFF):  # zeros, and all-ones bytes (a NaN in every float)
        ws = torch.full((need,), fill, dtype=torch.uint8, device="cuda")
        want = fa.bwd(x["q"], x["k"], x["v"], o, lse, x["dO"], 64, SCHED, layer0=15, workspace=ws)
        _assert_same(want, got)
    for g in got:
        assert torch.isfinite(g.float()).all()


def test_noalloc_at_its_size_limit_and_beyond():
    # the 16-layer training-step shape (B=8, H=8, T=1024) needs 32 MiB: it fits
    x = _inputs((16, 8, 8, 1024, 64), seed=43)
    assert fa.bwd_workspace_size(x["q"], 64, SCHED) <= fa.NOALLOC_SCRATCH_BYTES
    _compare(x)
    del x
    # twice the batch needs 64 MiB: rejected before any launch
    y = _inputs((16, 16, 8, 1024, 64), seed=44)
    assert fa.bwd_workspace_size(y["q"], 64, SCHED) > fa.NOALLOC_SCRATCH_BYTES
    o = torch.empty_like(y["q"])
    lse = torch.empty(y["q"].shape[:-1], dtype=torch.float32, device="cuda")
    with pytest.raises(fa.FibAttnError) as e:
        fa.bwd_noalloc(y["q"], y["k"], y["v"], o, lse, y["dO"], 64, SCHED)
    assert e.value.status == fa.SCRATCH_LIMIT
