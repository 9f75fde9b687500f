"""Pins of the oracle's grouped-query (GQA / MQA) wrappers (CPU only).

Query head h reads kv head h // G (H = G * H_kv). Checked against: the multi-head oracle at
G = 1, a per-head loop over the multi-head oracle, torch SDPA in fp64 with the kv heads
expanded by repeat_interleave and autograd for the gradients (a shared row's gradient is the
sum over the heads that read it), and central differences on shared rows.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import schedule as S


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def mask(T, W, tab):
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    m = (i - j >= 0) & (i - j < W)
    for o in tab:
        m |= (i - j) == o
    return torch.from_numpy(m)


@pytest.mark.parametrize("H,Hkv", [(4, 4), (4, 2), (8, 1), (6, 3)])
def test_gqa_matches_sdpa_and_autograd(H, Hkv):
    B, T, d, W = 2, 150, 16, 8
    tab = S.offset_table(S.FIB, Fraction(3, 2), W, T)
    q, g = rnd((B, H, T, d), 1), rnd((B, H, T, d), 4)
    k, v = rnd((B, Hkv, T, d), 2), rnd((B, Hkv, T, d), 3)
    scale = 1 / math.sqrt(d)
    out, lse = oracle.fwd_gqa(q, k, v, W, tab, scale)
    dq, dk, dv, out2, _ = oracle.bwd_gqa(q, k, v, g, W, tab, scale)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    G = H // Hkv
    ref = F.scaled_dot_product_attention(tq, tk.repeat_interleave(G, dim=-3),
                                         tv.repeat_interleave(G, dim=-3),
                                         attn_mask=mask(T, W, tab), scale=scale)
    (ref * torch.from_numpy(g)).sum().backward()
    np.testing.assert_allclose(out, ref.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(out2, out, rtol=0, atol=0)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-11)
    assert dk.shape == k.shape and dv.shape == v.shape


def test_gqa_per_head_loop_and_group_one():
    Lc, B, H, Hkv, T, d, W = 2, 1, 4, 2, 120, 8, 6
    tabs = [S.offset_table(S.FIB, Fraction(a), W, T) for a in (1, 2)]
    q = rnd((Lc, B, H, T, d), 5)
    k, v = rnd((Lc, B, Hkv, T, d), 6), rnd((Lc, B, Hkv, T, d), 7)
    out, lse = oracle.fwd_gqa(q, k, v, W, tabs)
    for l in range(Lc):
        for h in range(H):
            o1, l1 = oracle.fwd(q[l, :, h], k[l, :, h // 2], v[l, :, h // 2], W, tabs[l])
            np.testing.assert_array_equal(out[l, :, h], o1)
            np.testing.assert_array_equal(lse[l, :, h], l1)
    kk, vv = rnd((Lc, B, H, T, d), 8), rnd((Lc, B, H, T, d), 9)
    a = oracle.fwd_gqa(q, kk, vv, W, tabs)
    b = oracle.fwd(q, kk, vv, W, tabs)
    np.testing.assert_array_equal(a[0], b[0])


def test_gqa_central_differences_on_shared_rows():
    B, H, Hkv, T, d, W = 1, 4, 1, 90, 8, 5
    tab = S.offset_table(S.FIB, Fraction(1), W, T)
    q, g = rnd((B, H, T, d), 11), rnd((B, H, T, d), 12)
    k, v = rnd((B, Hkv, T, d), 13), rnd((B, Hkv, T, d), 14)
    _, dk, dv, _, _ = oracle.bwd_gqa(q, k, v, g, W, tab)
    loss = lambda k_, v_: float((g * oracle.fwd_gqa(q, k_, v_, W, tab)[0]).sum())
    h = 1e-6
    for (j, c) in ((10, 0), (55, 3), (89, 7), (0, 2)):
        for arr, grad, which in ((k, dk, "k"), (v, dv, "v")):
            a1, a2 = arr.copy(), arr.copy()
            a1[0, 0, j, c] += h
            a2[0, 0, j, c] -= h
            fd = ((loss(a1, v) - loss(a2, v)) if which == "k" else (loss(k, a1) - loss(k, a2))) / (2 * h)
            assert abs(fd - grad[0, 0, j, c]) <= 1e-6 * max(1.0, abs(fd)), (which, j, c)


def test_gqa_rejects_bad_groups():
    with pytest.raises(ValueError):
        oracle.fwd_gqa(rnd((1, 3, 8, 4), 0), rnd((1, 2, 8, 4), 1), rnd((1, 2, 8, 4), 2), 2, [])
