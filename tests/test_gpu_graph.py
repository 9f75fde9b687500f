"""The path inside a CUDA graph: a forward and backward captured on a stream and replayed.

Every launch of the library is a kernel on the caller's stream with its parameters (tensor
maps, offset tables) passed by value, so a training step can be captured once and replayed
without any per-step host work. The first call on a device sets per-kernel attributes and
caches device data, so it is made before the capture, as for any library that configures
kernels lazily. Replays must give the eager results bit for bit.
"""
import pytest
import torch

import fibattn_inputs as fi
import static_fibonacci_offset_fibattn_b300 as fa

pytestmark = pytest.mark.gpu


def test_training_step_captured_and_replayed_matches_eager():
    spec = fi.WORKLOADS["c5"]
    x = {n: t.cuda() for n, t in fi.workload_inputs("c5", layers=range(4), B=2).items()}
    sc = fa.Schedule(**spec["sched"])
    W = spec["W"]
    o = torch.empty_like(x["q"])
    lse = torch.empty(x["q"].shape[:-1], dtype=torch.float32, device="cuda")
    dq, dk, dv = (torch.empty_like(x[n]) for n in ("q", "k", "v"))
    ws = torch.empty(fa.bwd_workspace_size(x["q"], W, sc), dtype=torch.uint8, device="cuda")

    def step():
        fa.fwd(x["q"], x["k"], x["v"], W, sc, out=o, lse=lse)
        fa.bwd(x["q"], x["k"], x["v"], o, lse, x["dO"], W, sc, dq=dq, dk=dk, dv=dv, workspace=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # eager, outside the capture: the per-device first-call setup
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    want = [t.clone() for t in (o, lse, dq, dk, dv)]

    g = torch.cuda.CUDAGraph()
    for t in (o, lse, dq, dk, dv):
        t.zero_()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        for t in (o, lse, dq, dk, dv):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        fa.poll_device_error()
        for a, b in zip((o, lse, dq, dk, dv), want):
            assert torch.equal(a, b)
    # a replay reads the inputs' current contents: new inputs in the same buffers
    x["q"].mul_(0.5)
    g.replay()
    torch.cuda.synchronize()
    o2 = torch.empty_like(o)
    lse2 = torch.empty_like(lse)
    fa.fwd(x["q"], x["k"], x["v"], W, sc, out=o2, lse=lse2)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
