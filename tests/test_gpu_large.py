"""GPU parity at large sizes, where row, slice and tile indices get large: a 131,072-row
sequence (offsets up to 1974 rows back, 1024 tiles in one slice), 16,384 slices in one launch
(the TMA slice coordinate and the persistent tile walk), and the dense causal kernel at
T = 16,384 (128 key blocks for the last tile). Against the fp64 oracle, or against SDPA in fp32
where the oracle's O(T^2) cost is too high (needs a B300)."""
import numpy as np
import pytest
import torch

import fibattn_inputs as fi
import oracle
import static_fibonacci_offset_fibattn_b300 as fa
from gpu_common import (LSE_TOL, TOL, assert_grad, f64, lib_schedule, max_abs, oracle_table,
                        to_dev)

pytestmark = pytest.mark.gpu

STAGGER = dict(kind="linear", base="fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=16)


def test_long_sequence_fwd_bwd_matches_oracle():
    T, W, layer = 131072, 64, 15  # the top layer: alpha 2, offsets 68 .. 1974
    inp = fi.draw((1, 1, 1, T, 64), seed=301, scale=0.5, dtype="bf16", names=("q", "k", "v", "dO"))
    dev = to_dev(inp)
    sc = lib_schedule(STAGGER)
    tab = oracle_table(STAGGER, layer, W, T)
    assert fa.offsets(sc, layer, W, T) == tab and max(tab) > 1900
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], W, sc, layer0=layer)
    dq, dk, dv = fa.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["dO"], W, sc, layer0=layer)
    one = fa.bwd_fused(dev["q"], dev["k"], dev["v"], o, lse, dev["dO"], W, sc, layer0=layer)
    torch.cuda.synchronize()
    fa.poll_device_error()
    g = lambda n: f64(inp[n][0, 0, 0])
    rq, rk, rv, ro, rl = oracle.bwd(g("q"), g("k"), g("v"), g("dO"), W, tab)
    assert max_abs(f64(o[0, 0, 0]), ro) <= TOL["bf16"]
    assert max_abs(f64(lse[0, 0, 0]), rl) <= LSE_TOL["bf16"]
    for n, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert_grad(n, f64(got[0, 0, 0]), ref, "bf16")
    for a, b in zip(one, (dq, dk, dv)):
        assert torch.equal(a, b)


def test_many_slices_in_one_launch():
    # 16,384 (batch, head) slices of 128 rows: sampled slices across the whole range
    B, H, T, W, layer = 256, 64, 128, 16, 9
    inp = fi.draw((1, B, H, T, 64), seed=303, scale=0.5, dtype="bf16", names=("q", "k", "v", "dO"))
    dev = to_dev(inp)
    sc = lib_schedule(STAGGER)
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], W, sc, layer0=layer)
    dq, dk, dv = fa.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["dO"], W, sc, layer0=layer)
    torch.cuda.synchronize()
    fa.poll_device_error()
    tab = oracle_table(STAGGER, layer, W, T)
    picks = [(0, 0), (0, 63), (17, 5), (128, 32), (255, 0), (255, 63)]
    g = lambda n: np.stack([f64(inp[n][0, b, h]) for b, h in picks])
    rq, rk, rv, ro, rl = oracle.bwd(g("q"), g("k"), g("v"), g("dO"), W, tab)
    for idx, (b, h) in enumerate(picks):
        assert max_abs(f64(o[0, b, h]), ro[idx]) <= TOL["bf16"]
        assert max_abs(f64(lse[0, b, h]), rl[idx]) <= LSE_TOL["bf16"]
        for n, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
            assert_grad(n, f64(got[0, b, h]), ref[idx], "bf16", (b, h))


def test_dense_kernel_at_long_length_matches_sdpa():
    T = 16384
    dev = to_dev(fi.draw((1, 1, 2, T, 64), seed=305, scale=0.5, dtype="bf16"))
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], T, lib_schedule(STAGGER))
    torch.cuda.synchronize()
    fa.poll_device_error()
    q, k, v = (dev[n][0, 0].float() for n in "qkv")  # [2 heads, T, 64]
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    assert max_abs(f64(o[0, 0]), f64(ref)) <= TOL["bf16"]
    # lse of the last rows (the longest sums): exact from the fp32 scores
    s = (q[:, -256:] @ k.transpose(-1, -2)) * 0.125
    mask = torch.arange(T, device=s.device)[None, :] > torch.arange(T - 256, T, device=s.device)[:, None]
    s = s.masked_fill(mask, float("-inf"))
    assert max_abs(f64(lse[0, 0][:, -256:]), f64(torch.logsumexp(s, dim=-1))) <= LSE_TOL["bf16"]


def test_fp32_path_at_long_length():
    # the fp32 SIMT path (1e-5) on an 8,192-row sequence with offsets up to 1974 rows back
    T, W, layer = 8192, 64, 15
    inp = fi.draw((1, 1, 2, T, 64), seed=307, scale=0.5, dtype="f32", names=("q", "k", "v", "dO"))
    dev = to_dev(inp)
    sc = lib_schedule(STAGGER)
    o, lse = fa.fwd(dev["q"], dev["k"], dev["v"], W, sc, layer0=layer)
    dq, dk, dv = fa.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["dO"], W, sc, layer0=layer)
    torch.cuda.synchronize()
    fa.poll_device_error()
    tab = oracle_table(STAGGER, layer, W, T)
    g = lambda n: f64(inp[n][0, 0])
    rq, rk, rv, ro, rl = oracle.bwd(g("q"), g("k"), g("v"), g("dO"), W, tab)
    assert max_abs(f64(o[0, 0]), ro) <= TOL["f32"]
    assert max_abs(f64(lse[0, 0]), rl) <= LSE_TOL["f32"]
    for n, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert_grad(n, f64(got[0, 0]), ref, "f32")
