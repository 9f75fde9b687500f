"""Pins of the oracle's forward and backward attention (CPU only).

The oracle (C, fp64, materialised key lists) is checked against things it does not
share code with: torch's scaled_dot_product_attention in fp64 with a mask built
by brute force from the key-set predicate, its dense-causal and sliding-window
special cases, closed forms (V = 1, Q = 0, first query), softmax shift invariance,
central finite differences and autograd.
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
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) * scale


def bf_mask(T, W, tab):
    """Boolean [T, T] mask by brute force: key j allowed for query i iff
    0 <= i - j < W or i - j is in the table."""
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    dist = i - j
    m = (dist >= 0) & (dist < W)
    for o in tab:
        m |= dist == o
    return torch.from_numpy(m)


def sdpa(q, k, v, mask, scale):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    return F.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=mask, scale=scale).numpy()


def lse_ref(q, k, mask, scale):
    s = torch.from_numpy(q) @ torch.from_numpy(k).transpose(-1, -2) * scale
    s = s.masked_fill(~mask, -math.inf)
    return torch.logsumexp(s, dim=-1).numpy()


CASES = [
    # (B, H, T, d, W, base, alpha)
    (1, 2, 256, 64, 16, S.FIB, Fraction(1)),
    (2, 1, 300, 16, 12, S.FIB, Fraction(3, 2)),
    (1, 2, 129, 8, 6, S.POW2, Fraction(1)),
    (1, 1, 200, 32, 8, S.FIB, Fraction(1, 2)),
    (1, 1, 1, 8, 4, S.FIB, Fraction(1)),
]


@pytest.mark.parametrize("case", CASES)
def test_fwd_matches_library_masked_attention(case):
    B, H, T, d, W, base, alpha = case
    tab = S.offset_table(base, alpha, W, T)
    q, k, v = (rnd((B, H, T, d), s) for s in (1, 2, 3))
    scale = 1 / math.sqrt(d)
    out, lse = oracle.fwd(q, k, v, W, tab, scale)
    m = bf_mask(T, W, tab)
    np.testing.assert_allclose(out, sdpa(q, k, v, m, scale), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref(q, k, m, scale), rtol=0, atol=1e-12)


def test_fwd_dense_causal_when_window_covers_sequence():
    T, d = 97, 16
    q, k, v = (rnd((1, 3, T, d), s) for s in (4, 5, 6))
    t = lambda a: torch.from_numpy(a)
    ref = F.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True).numpy()
    for W in (T, T + 5, 10 ** 6):
        out, _ = oracle.fwd(q, k, v, W, [], None)
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_fwd_sliding_window_when_table_empty():
    T, d, W = 150, 16, 20
    q, k, v = (rnd((2, 1, T, d), s) for s in (7, 8, 9))
    # base_max below the window: no offsets survive
    tab = S.offset_table(S.FIB, Fraction(1), W, T, base_max=W - 1)
    assert tab == []
    band = torch.ones(T, T, dtype=torch.bool).tril() & ~torch.ones(T, T, dtype=torch.bool).tril(-W)
    out, _ = oracle.fwd(q, k, v, W, tab, None)
    np.testing.assert_allclose(out, sdpa(q, k, v, band, 1 / math.sqrt(d)), rtol=0, atol=1e-12)


def test_fwd_closed_forms():
    T, d, W = 180, 8, 10
    tab = S.offset_table(S.FIB, Fraction(1), W, T)
    q, k, v = (rnd((1, 1, T, d), s) for s in (10, 11, 12))
    # V = 1: every output row is exactly 1 (softmax rows sum to one)
    out, _ = oracle.fwd(q, k, np.ones_like(v), W, tab)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-13)
    # Q = 0: uniform weights, O_i = mean of V over S_i, LSE_i = ln |S_i|
    out, lse = oracle.fwd(np.zeros_like(q), k, v, W, tab)
    for i in range(T):
        n = min(W, i + 1) + sum(1 for o in tab if o <= i)
        js = [j for j in range(T) if 0 <= i - j < W or (i - j) in tab]
        assert len(js) == n
        np.testing.assert_allclose(out[0, 0, i], v[0, 0, js].mean(0), rtol=0, atol=1e-13)
        assert abs(lse[0, 0, i] - math.log(n)) < 1e-13
    # first query sees only itself
    out, lse = oracle.fwd(q, k, v, W, tab)
    np.testing.assert_allclose(out[0, 0, 0], v[0, 0, 0], rtol=0, atol=1e-15)
    assert abs(lse[0, 0, 0] - float(q[0, 0, 0] @ k[0, 0, 0]) / math.sqrt(d)) < 1e-13


def test_fwd_shift_invariance():
    # adding one vector c to every key adds scale*q_i.c to every score of row i:
    # outputs unchanged, lse shifted by that amount
    T, d, W = 120, 16, 8
    tab = S.offset_table(S.FIB, Fraction(3, 2), W, T)
    q, k, v = (rnd((1, 2, T, d), s) for s in (13, 14, 15))
    c = rnd((d,), 16)
    o1, l1 = oracle.fwd(q, k, v, W, tab)
    o2, l2 = oracle.fwd(q, k + c, v, W, tab)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1 + (q @ c) / math.sqrt(d), rtol=0, atol=1e-12)


def test_fwd_per_layer_tables():
    # a leading layer axis with a table per layer equals per-layer calls
    L, T, d, W = 3, 160, 8, 8
    tabs = [S.layer_table(S.FIB, S.LINEAR, l, L, W, T) for l in range(L)]
    q, k, v = (rnd((L, 2, 1, T, d), s) for s in (17, 18, 19))
    out, lse = oracle.fwd(q, k, v, W, tabs)
    for l in range(L):
        o1, l1 = oracle.fwd(q[l], k[l], v[l], W, tabs[l])
        np.testing.assert_array_equal(out[l], o1)
        np.testing.assert_array_equal(lse[l], l1)


def _loss(q, k, v, g, W, tab):
    out, _ = oracle.fwd(q, k, v, W, tab)
    return float((out * g).sum())


def test_bwd_central_finite_differences():
    T, d, W = 40, 6, 5
    tab = S.offset_table(S.FIB, Fraction(1), W, T)
    q, k, v, g = (rnd((1, 1, T, d), s) for s in (20, 21, 22, 23))
    dq, dk, dv, _, _ = oracle.bwd(q, k, v, g, W, tab)
    h = 1e-6
    rng = np.random.default_rng(0)
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(25):
            idx = (0, 0, int(rng.integers(T)), int(rng.integers(d)))
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            fp = _loss(*(xp if n == name else args[n] for n in "qkv"), g, W, tab)
            fm = _loss(*(xm if n == name else args[n] for n in "qkv"), g, W, tab)
            num = (fp - fm) / (2 * h)
            assert abs(num - grad[idx]) <= 1e-6 * max(1.0, abs(num)), (name, idx, num, grad[idx])


@pytest.mark.parametrize("case", CASES[:4])
def test_bwd_matches_autograd(case):
    B, H, T, d, W, base, alpha = case
    tab = S.offset_table(base, alpha, W, T)
    q, k, v, g = (rnd((B, H, T, d), s) for s in (24, 25, 26, 27))
    scale = 1 / math.sqrt(d)
    dq, dk, dv, out, lse = oracle.bwd(q, k, v, g, W, tab, scale)
    tq, tk, tv = (torch.from_numpy(a.copy()).requires_grad_() for a in (q, k, v))
    ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=bf_mask(T, W, tab), scale=scale)
    ref.backward(torch.from_numpy(g))
    np.testing.assert_allclose(out, ref.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-11)


def test_bwd_gradient_sums():
    # sum_i dQ_i . q_i ... simpler invariant: V = 1 makes dS = 0, so dQ = dK = 0;
    # and dV sums, over keys, to the sum of dO (each row's weights sum to one)
    T, d, W = 90, 8, 7
    tab = S.offset_table(S.FIB, Fraction(1), W, T)
    q, k, g = (rnd((1, 1, T, d), s) for s in (28, 29, 30))
    dq, dk, dv, _, _ = oracle.bwd(q, k, np.ones_like(q), g, W, tab)
    np.testing.assert_allclose(dq, 0, atol=1e-13)
    np.testing.assert_allclose(dk, 0, atol=1e-13)
    np.testing.assert_allclose(dv.sum(2), g.sum(2), rtol=0, atol=1e-12)
