"""GPU tests of fibattn_fwd_bwd: the forward and backward of a layer stack with the layers
split into groups on concurrent streams. Its outputs must equal fwd() followed by bwd() bit
for bit (the same kernels on the same inputs, each group on its own workspace), for every
number of streams, head layout and dtype, and inside a captured CUDA graph (needs a B300)."""
import pytest
import torch

import fibattn_inputs as fi
import static_fibonacci_offset_fibattn_b300 as fa
from gpu_common import lib_schedule, to_dev

pytestmark = pytest.mark.gpu

SCHED = dict(kind="coprime", base="fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=16,
             coprime_c=5)


def _sequential(dev, W, sc, layer0):
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], W, sc, layer0=layer0)
    dq, dk, dv = fa.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["dO"], W, sc, layer0=layer0)
    return o, lse, dq, dk, dv


def _assert_same(a, b):
    for n, x, y in zip(("o", "lse", "dq", "dk", "dv"), a, b):
        assert torch.equal(x, y), n


@pytest.mark.parametrize("n_streams", [1, 2, 3, 4, 8])
def test_fwd_bwd_equals_sequential_calls(n_streams):
    inp = to_dev(fi.draw((6, 2, 4, 700, 64), seed=91, scale=0.5, dtype="bf16",
                         names=("q", "k", "v", "dO")))
    sc = lib_schedule(SCHED)
    got = fa.fwd_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], 64, sc, layer0=3,
                     n_streams=n_streams)
    want = _sequential(inp, 64, sc, 3)
    torch.cuda.synchronize()
    fa.poll_device_error()
    _assert_same(got, want)


@pytest.mark.parametrize("case", [("bf16", 64, 8, 2), ("bf16", 128, 4, 4), ("f32", 64, 2, 2)])
def test_fwd_bwd_head_layouts_and_dtypes(case):
    dtype, d, H, Hkv = case
    kv = {n: (5, 1, Hkv, 300, d) for n in ("k", "v")}
    inp = to_dev(fi.draw((5, 1, H, 300, d), seed=93, scale=0.5, dtype=dtype,
                         names=("q", "k", "v", "dO"), shapes=kv))
    sc = lib_schedule(SCHED)
    got = fa.fwd_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], 16, sc, n_streams=2)
    want = _sequential(inp, 16, sc, 0)
    torch.cuda.synchronize()
    _assert_same(got, want)


def test_fwd_bwd_training_step_and_graph_capture():
    # the full training-step shape (16 layers x B8 H8 T1024) on two streams, eager and as a
    # captured graph replayed after the inputs change
    spec = fi.WORKLOADS["c5"]
    inp = to_dev(fi.workload_inputs("c5"))
    sc = lib_schedule(spec["sched"])
    want = _sequential(inp, 64, sc, 0)
    outs = [torch.empty_like(t) for t in want]
    ws = torch.empty(fa.fwd_bwd_workspace_size(inp["q"], 64, sc, n_streams=2), dtype=torch.uint8,
                     device="cuda")
    step = lambda: fa.fwd_bwd(inp["q"], inp["k"], inp["v"], inp["dO"], 64, sc, n_streams=2,
                              out=outs[0], lse=outs[1], dq=outs[2], dk=outs[3], dv=outs[4],
                              workspace=ws)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    _assert_same(outs, want)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    inp["dO"].mul_(2)  # a new upstream gradient: the replay must see it
    want2 = _sequential(inp, 64, sc, 0)
    for t in outs:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    fa.poll_device_error()
    _assert_same(outs, want2)
