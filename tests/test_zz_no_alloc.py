"""fibattn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: an operator hosted by a framework that owns the
device allocator and passes it no workspace, or a latency-critical loop where
cudaMalloc/cudaFree would synchronise the device. fibattn_bwd needs a caller-allocated
workspace (D per row and the (P, dS) pair of every diagonal entry); fibattn_bwd_noalloc
takes it from a fixed 40 MiB per-device array inside the library instead. These tests call it through the C ABI, twice
in a row (the array keeps the previous call's contents), and compare it with fibattn_bwd
within the bf16 tolerance the parity tests use.

This file is collected last on purpose, so that a run stopping at its first failure has
already run every other test.
"""
import pytest
import torch

import fibattn_inputs as fi
import static_fibonacci_offset_fibattn_b300 as fa
from gpu_common import TOL, f64, max_abs

pytestmark = pytest.mark.gpu

SCHED = fa.Schedule("coprime", "fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=16, coprime_c=5)


def _inputs(shape, seed):
    inp = fi.draw(shape, seed=seed, scale=0.125, dtype="bf16", names=("q", "k", "v", "dO"))
    return {n: t.cuda() for n, t in inp.items()}


def _compare(x, layer0=0):
    o, lse = fa.fwd(x["q"], x["k"], x["v"], 64, SCHED, layer0=layer0)
    want = fa.bwd(x["q"], x["k"], x["v"], o, lse, x["dO"], 64, SCHED, layer0=layer0)
    got = fa.bwd_noalloc(x["q"], x["k"], x["v"], o, lse, x["dO"], 64, SCHED, layer0=layer0)
    torch.cuda.synchronize()
    fa.poll_device_error()
    for name, a, b in zip(("dq", "dk", "dv"), want, got):
        err = max_abs(f64(a), f64(b))
        assert err <= TOL["bf16"], (name, err)


def test_noalloc_matches_bwd_on_two_calls_in_a_row():
    # two different inputs back to back: the second call must not see the first's workspace
    _compare(_inputs((2, 2, 4, 1024, 64), seed=41), layer0=3)
    _compare(_inputs((3, 1, 2, 777, 64), seed=42), layer0=9)


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
