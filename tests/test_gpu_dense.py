"""GPU parity of the dense causal forward (the W >= T case: no offset survives the table rule,
every earlier key is attended), which fibattn_fwd runs on its own tensor-core kernel at bf16
and head size 64. Against the fp64 oracle (max-abs 2e-2 on o, 1e-3 on lse), on ragged tails,
grouped-query heads, several layers per call and inputs large enough that the running max
is raised (and O rescaled) between key blocks (needs a B300)."""
import pytest
import torch

import fibattn_inputs as fi
import oracle
import static_fibonacci_offset_fibattn_b300 as fa
from gpu_common import LSE_TOL, TOL, f64, lib_schedule, max_abs, oracle_table, to_dev

pytestmark = pytest.mark.gpu

SCHED = dict(kind="linear", base="fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=16)

DENSE = [
    # (Lc, B, H, Hkv, T, W, scale)
    (1, 1, 2, 2, 1, 1, 0.5),        # one row
    (1, 1, 2, 2, 127, 127, 0.5),    # one partial tile
    (1, 2, 2, 2, 128, 128, 0.5),    # one full tile
    (1, 1, 3, 3, 129, 200, 0.5),    # a last tile of one row; W > T
    (2, 1, 4, 2, 300, 300, 0.5),    # two layers in one call, grouped-query heads
    (1, 1, 4, 1, 640, 640, 0.5),    # multi-query: one kv head
    (1, 1, 2, 2, 1000, 4096, 2.0),  # large scores (q, k at scale 2, v at 1/4): the running max
                                    # rises past 2^8 between key blocks, O is rescaled in TMEM
]


@pytest.mark.parametrize("case", DENSE)
def test_dense_forward_matches_oracle(case):
    Lc, B, H, Hkv, T, W, scale = case
    layer0 = 5
    kv = {n: (Lc, B, Hkv, T, 64) for n in ("k", "v")}
    inp = fi.draw((Lc, B, H, T, 64), seed=500 + T, scale=scale, dtype="bf16", shapes=kv)
    # v drawn on its own at scale 1/4 when q and k are large, so that o stays where bf16's
    # spacing is below the 2e-2 bound (53 (row, block) pairs of the stress case raise the max)
    if scale > 0.5:
        inp["v"] = fi.draw((Lc, B, Hkv, T, 64), seed=900 + T, scale=0.25, dtype="bf16",
                           names=("v",))["v"]
    sc = lib_schedule(SCHED)
    assert all(fa.offsets(sc, layer0 + l, W, T) == [] for l in range(Lc))
    dev = to_dev(inp)
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], W, sc, layer0=layer0)
    torch.cuda.synchronize()
    fa.poll_device_error()
    tabs = [oracle_table(SCHED, layer0 + l, W, T) for l in range(Lc)]
    ro, rl = oracle.fwd_gqa(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), W, tabs)
    assert max_abs(f64(o), ro) <= TOL["bf16"]
    assert max_abs(f64(lse), rl) <= LSE_TOL["bf16"]


def test_dense_forward_matches_sdpa_at_4x_length_all_slices():
    # one layer of the 4x-length inputs (B2 H8 T4096): every slice against SDPA in fp32
    spec = fi.WORKLOADS["c4"]
    dev = to_dev(fi.workload_inputs("c4", layers=[0]))
    T = spec["T"]
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], T, lib_schedule(spec["sched"]))
    q, k, v = (dev[n][0].float() for n in "qkv")
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    s = (q @ k.transpose(-1, -2)) * 0.125
    s = s.masked_fill(torch.ones(T, T, dtype=torch.bool, device=s.device).triu(1), float("-inf"))
    assert max_abs(f64(o[0]), f64(ref)) <= TOL["bf16"]
    assert max_abs(f64(lse[0]), f64(torch.logsumexp(s, dim=-1))) <= LSE_TOL["bf16"]


def test_dense_forward_deterministic_and_backward_consistent():
    # repeated calls give the same bits, and the backward from the dense forward's o and lse
    # matches the oracle's gradient of dense causal attention
    inp = fi.draw((1, 1, 2, 515, 64), seed=77, scale=0.5, dtype="bf16", names=("q", "k", "v", "dO"))
    dev = to_dev(inp)
    sc = lib_schedule(SCHED)
    a = fa.fwd(dev["q"], dev["k"], dev["v"], 515, sc)
    b = fa.fwd(dev["q"], dev["k"], dev["v"], 515, sc)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    dq, dk, dv = fa.bwd(dev["q"], dev["k"], dev["v"], a[0], a[1], dev["dO"], 515, sc)
    torch.cuda.synchronize()
    tab = oracle_table(SCHED, 0, 515, 515)
    rq, rk, rv, ro, rl = oracle.bwd(f64(inp["q"][0]), f64(inp["k"][0]), f64(inp["v"][0]),
                                    f64(inp["dO"][0]), 515, tab)
    from gpu_common import assert_grad
    for n, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert_grad(n, f64(got[0]), ref, "bf16")


def test_dense_forward_more_layers_than_one_launch():
    # 18 layers (launches of 16 + 2) equal the per-layer calls bit for bit
    sched = dict(kind="linear", base="fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=20)
    sc = lib_schedule(sched)
    dev = to_dev(fi.draw((18, 1, 2, 333, 64), seed=79, scale=0.5, dtype="bf16"))
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], 400, sc, layer0=1)
    for c in (0, 15, 16, 17):
        oc, lc = fa.fwd(dev["q"][c], dev["k"][c], dev["v"][c], 400, sc, layer0=1 + c)
        assert torch.equal(oc, o[c]) and torch.equal(lc, lse[c])
