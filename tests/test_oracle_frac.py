"""Pins of the oracle's fractional-offset forward (CPU only).

The learned-alpha variant interpolates keys and values linearly between the two rows
around the real position i - alpha * F ("Depth-Staggered Fibonacci Spacing for Sparse
Attention", gist.science explainer, Metodologia / Arquitetura, "Implementacao"). The
oracle's per-query loop is checked against: the static oracle at integer distances, a
vectorised torch fp64 formulation with gathered interpolated rows, closed forms for keys
and values that are linear in the position (interpolation of a linear function is exact),
continuity in alpha across integer distances, and the distance list rule.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import schedule as S


def rnd(shape, seed, scale=1.0):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) * scale


def f32(a):
    """alpha as the float32 value the library receives."""
    return float(np.float32(a))


def torch_frac_fwd(q, k, v, W, dists, scale):
    """Vectorised fp64 statement: window scores from a masked q k^T, one gathered and
    interpolated key/value row per (query, distance), softmax over the concatenation."""
    q, k, v = (torch.from_numpy(np.ascontiguousarray(a)) for a in (q, k, v))
    T = q.shape[-2]
    i = torch.arange(T, dtype=torch.float64)
    dist = i[:, None] - i[None, :]
    win = (dist >= 0) & (dist < W)
    s_win = (q @ k.transpose(-1, -2) * scale).masked_fill(~win, -math.inf)
    s_parts, v_parts = [s_win], []
    for dk in dists:
        pos = i - dk
        ok = pos >= 0
        lo = torch.floor(pos).clamp(min=0).long()
        w = (pos - torch.floor(pos)).clamp(min=0)
        hi = (lo + 1).clamp(max=T - 1)
        kt = (1 - w)[:, None] * k[..., lo, :] + w[:, None] * k[..., hi, :]
        vt = (1 - w)[:, None] * v[..., lo, :] + w[:, None] * v[..., hi, :]
        s = (q * kt).sum(-1) * scale
        s_parts.append(s.masked_fill(~ok, -math.inf)[..., None])
        v_parts.append(vt)
    s_all = torch.cat(s_parts, dim=-1)
    lse = torch.logsumexp(s_all, dim=-1)
    p = torch.exp(s_all - lse[..., None])
    out = p[..., :T] @ v
    for t, vt in enumerate(v_parts):
        out = out + p[..., T + t, None] * vt
    return out.numpy(), lse.numpy()


def positions(i, W, dists):
    """Real positions attended by query i: its window rows and every i - d >= 0."""
    pos = [float(j) for j in range(max(0, i - W + 1), i + 1)]
    pos += [i - dk for dk in dists if i - dk >= 0]
    return np.array(pos)


@pytest.mark.parametrize("alpha,base,W,T", [(1.0, S.FIB, 16, 256), (2.0, S.FIB, 8, 300),
                                            (3.0, S.POW2, 4, 200), (1.0, S.POW2, 1, 64)])
def test_integer_alpha_reduces_to_static_oracle(alpha, base, W, T):
    dists = oracle.frac_distances(alpha, base, W, T)
    tab = S.offset_table(base, Fraction(alpha), W, T)
    assert dists == [float(o) for o in tab]
    q, k, v = (rnd((2, T, 32), s) for s in (1, 2, 3))
    out_f, lse_f = oracle.fwd_frac(q, k, v, W, dists)
    out_s, lse_s = oracle.fwd(q, k, v, W, tab)
    np.testing.assert_allclose(out_f, out_s, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse_f, lse_s, rtol=0, atol=1e-13)


@pytest.mark.parametrize("alpha,base,W,T,d", [(1.37, S.FIB, 16, 256, 32), (0.61, S.FIB, 3, 130, 16),
                                              (2.718, S.POW2, 5, 300, 8), (0.5, S.FIB, 1, 90, 8)])
def test_matches_vectorised_gather(alpha, base, W, T, d):
    dists = oracle.frac_distances(f32(alpha), base, W, T)
    assert any(dk != math.floor(dk) for dk in dists)
    q, k, v = (rnd((1, 2, T, d), s) for s in (4, 5, 6))
    scale = 1 / math.sqrt(d)
    out, lse = oracle.fwd_frac(q, k, v, W, dists, scale)
    ro, rl = torch_frac_fwd(q, k, v, W, dists, scale)
    np.testing.assert_allclose(out, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rl, rtol=0, atol=1e-12)


def test_uniform_attention_over_linear_values():
    # q = 0: every attended key weighs the same; v_j = a + b j, so the interpolated value
    # at real position p is a + b p and o_i = a + b * mean(attended positions).
    T, d, W = 200, 8, 6
    dists = oracle.frac_distances(f32(1.23), S.FIB, W, T)
    a, b = rnd(d, 7), rnd(d, 8)
    v = a[None, :] + np.arange(T)[:, None] * b[None, :]
    q = np.zeros((T, d))
    k = rnd((T, d), 9)
    out, lse = oracle.fwd_frac(q, k, v, W, dists)
    for i in range(T):
        pos = positions(i, W, dists)
        np.testing.assert_allclose(out[i], a + b * pos.mean(), rtol=0, atol=1e-10)
        assert abs(lse[i] - math.log(len(pos))) < 1e-12


def test_linear_keys_give_scores_linear_in_position():
    # k_j = a + b j: the interpolated key at p is a + b p, its score scale q.(a + b p).
    T, d, W = 160, 16, 4
    dists = oracle.frac_distances(f32(0.77), S.FIB, W, T)
    a, b = rnd(d, 10), rnd(d, 11, 0.05)
    k = a[None, :] + np.arange(T)[:, None] * b[None, :]
    v = a[None, :] * 0.5 + np.arange(T)[:, None] * b[None, :] * 2.0
    q = rnd((T, d), 12)
    scale = 0.25
    out, lse = oracle.fwd_frac(q, k, v, W, dists, scale)
    for i in range(T):
        pos = positions(i, W, dists)
        s = scale * (q[i] @ a + (q[i] @ b) * pos)
        m = s.max()
        p = np.exp(s - m)
        l = p.sum()
        exp_o = 0.5 * a + 2.0 * b * float((p * pos).sum() / l)
        np.testing.assert_allclose(out[i], exp_o, rtol=0, atol=1e-10)
        assert abs(lse[i] - (m + math.log(l))) < 1e-12


@pytest.mark.parametrize("alpha", [1.0, 2.0])
def test_continuous_in_alpha_across_integer_distances(alpha):
    # Linear interpolation is continuous in the position: nudging alpha across an integer
    # moves the output by O(eps), from either side. (W is no multiple of alpha F, so no
    # distance enters or leaves the kept interval W <= d <= T - 1.) The rows i = d are
    # left out: there the interpolated key sits at position 0 and, by the causal rule, it
    # exists only for i - d >= 0.
    T, d, W = 180, 16, 7
    q, k, v = (rnd((T, d), s) for s in (13, 14, 15))
    d0 = oracle.frac_distances(alpha, S.FIB, W, T)
    ref, _ = oracle.fwd_frac(q, k, v, W, d0)
    rows = [i for i in range(T) if float(i) not in d0]
    for eps in (1e-7, -1e-7):
        da = oracle.frac_distances(alpha + eps, S.FIB, W, T)
        assert len(da) == len(d0)
        out, _ = oracle.fwd_frac(q, k, v, W, da)
        diff = np.abs(out - ref)
        assert 0 < diff[rows].max() < 1e-4
        if eps > 0:  # d just above i: the key at position 0 drops out (a jump)
            assert diff[[int(x) for x in d0]].max() > 1e-2


def test_distance_list_rule():
    # d = alpha F in double from the float32 alpha, kept when W <= d <= T - 1
    alpha = f32(1.37)
    fib = [1, 2, 3, 5, 8, 13, 21, 34, 55, 89, 144, 233, 377, 610, 987]
    want = [alpha * f for f in fib if 16 <= alpha * f <= 255]
    assert oracle.frac_distances(alpha, S.FIB, 16, 256) == want
    assert oracle.frac_distances(alpha, S.FIB, 16, 256, base_max=100) == [x for x in want if x <= alpha * 100]
    pw = [alpha * 2 ** e for e in range(12) if 5 <= alpha * 2 ** e <= 299]
    assert oracle.frac_distances(alpha, S.POW2, 5, 300) == pw
    with pytest.raises(ValueError):
        oracle.frac_distances(0.0, S.FIB, 4, 10)


def test_per_layer_distance_lists():
    T, d, W = 140, 8, 4
    q, k, v = (rnd((2, 1, 2, T, d), s) for s in (16, 17, 18))
    tabs = [oracle.frac_distances(f32(a), S.FIB, W, T) for a in (0.9, 1.6)]
    out, lse = oracle.fwd_frac(q, k, v, W, tabs)
    for l in range(2):
        o1, l1 = oracle.fwd_frac(q[l], k[l], v[l], W, tabs[l])
        np.testing.assert_array_equal(out[l], o1)
        np.testing.assert_array_equal(lse[l], l1)


# ------------------------------------------------------------------ backward


def torch_frac_loss(q, k, v, dout, W, alpha, bases, scale):
    """Sum(dout * out) of the vectorised statement, with alpha a leaf tensor: the position
    i - alpha F is split into a detached floor and a weight that carries the gradient."""
    T = q.shape[-2]
    i = torch.arange(T, dtype=torch.float64)
    dist = i[:, None] - i[None, :]
    win = (dist >= 0) & (dist < W)
    s_parts = [(q @ k.transpose(-1, -2) * scale).masked_fill(~win, -math.inf)]
    v_parts = []
    for f in bases:
        pos = i - alpha * f
        ok = pos.detach() >= 0
        lo = torch.floor(pos.detach()).clamp(min=0)
        w = torch.where(ok, pos - lo, torch.zeros_like(pos))
        lo = lo.long()
        hi = (lo + 1).clamp(max=T - 1)
        kt = (1 - w)[:, None] * k[..., lo, :] + w[:, None] * k[..., hi, :]
        vt = (1 - w)[:, None] * v[..., lo, :] + w[:, None] * v[..., hi, :]
        s = (q * kt).sum(-1) * scale
        s_parts.append(s.masked_fill(~ok, -math.inf)[..., None])
        v_parts.append(vt)
    s_all = torch.cat(s_parts, dim=-1)
    p = torch.softmax(s_all, dim=-1)
    out = p[..., :T] @ v
    for t, vt in enumerate(v_parts):
        out = out + p[..., T + t, None] * vt
    return (dout * out).sum()


@pytest.mark.parametrize("alpha,base,W,T,d", [(1.37, S.FIB, 16, 256, 16), (0.61, S.FIB, 3, 130, 8),
                                              (2.718, S.POW2, 5, 300, 8), (1.0, S.FIB, 8, 200, 8)])
def test_bwd_frac_matches_autograd(alpha, base, W, T, d):
    a = f32(alpha)
    dists = oracle.frac_distances(a, base, W, T)
    bases = oracle.frac_bases(a, base, W, T)
    assert [a * f for f in bases] == dists
    q, k, v, g = (rnd((2, T, d), s) for s in (21, 22, 23, 24))
    scale = 1 / math.sqrt(d)
    dq, dk, dv, out, lse, dd = oracle.bwd_frac(q, k, v, g, W, dists, scale)
    t = [torch.tensor(x, requires_grad=True) for x in (q, k, v)]
    at = torch.tensor(a, dtype=torch.float64, requires_grad=True)
    loss = torch_frac_loss(*t, torch.from_numpy(g), W, at, bases, scale)
    loss.backward()
    np.testing.assert_allclose(dq, t[0].grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, t[1].grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, t[2].grad.numpy(), rtol=0, atol=1e-11)
    dalpha = float((dd[:, : len(bases)] * np.array(bases, dtype=np.float64)).sum())
    assert abs(dalpha - at.grad.item()) <= 1e-9 * max(1.0, abs(dalpha))


def test_bwd_frac_central_differences():
    T, d, W, alpha = 150, 8, 6, f32(1.37)
    q, k, v, g = (rnd((T, d), s) for s in (31, 32, 33, 34))
    dists = oracle.frac_distances(alpha, S.FIB, W, T)
    bases = oracle.frac_bases(alpha, S.FIB, W, T)
    dq, dk, dv, _, _, dd = oracle.bwd_frac(q, k, v, g, W, dists)
    loss = lambda q_, k_, v_, ds: float((g * oracle.fwd_frac(q_, k_, v_, W, ds)[0]).sum())
    h = 1e-6
    # alpha: no distance is within h * F of an integer, so the segment stays the same
    assert all(min(x - math.floor(x), math.ceil(x) - x) > 1e-3 for x in dists)
    up = [(alpha + h) * f for f in bases]
    dn = [(alpha - h) * f for f in bases]
    fd = (loss(q, k, v, up) - loss(q, k, v, dn)) / (2 * h)
    dalpha = float((dd[: len(bases)] * np.array(bases, dtype=np.float64)).sum())
    assert abs(fd - dalpha) <= 1e-6 * max(1.0, abs(dalpha))
    # each distance on its own
    for t in range(len(dists)):
        up = list(dists); up[t] += h
        dn = list(dists); dn[t] -= h
        fd = (loss(q, k, v, up) - loss(q, k, v, dn)) / (2 * h)
        assert abs(fd - dd[t]) <= 1e-6 * max(1.0, abs(dd[t])), t
    # a few entries of q, k, v, among them rows that only an interpolated key reaches
    lo = int(math.floor(100 - dists[2]))
    for name, arr, grad, idx in (("q", q, dq, (100, 3)), ("k", k, dk, (lo, 5)),
                                 ("k", k, dk, (lo + 1, 0)), ("v", v, dv, (lo, 2)),
                                 ("v", v, dv, (lo + 1, 7)), ("k", k, dk, (140, 1))):
        a1, a2 = arr.copy(), arr.copy()
        a1[idx] += h
        a2[idx] -= h
        args1 = [a1 if n == name else x for n, x in (("q", q), ("k", k), ("v", v))]
        args2 = [a2 if n == name else x for n, x in (("q", q), ("k", k), ("v", v))]
        fd = (loss(*args1, dists) - loss(*args2, dists)) / (2 * h)
        assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(grad[idx])), (name, idx)


@pytest.mark.parametrize("alpha,base", [(1.0, S.FIB), (2.0, S.POW2)])
def test_bwd_frac_integer_alpha_reduces_to_static(alpha, base):
    T, d, W = 220, 16, 10
    q, k, v, g = (rnd((2, T, d), s) for s in (41, 42, 43, 44))
    dists = oracle.frac_distances(alpha, base, W, T)
    dq, dk, dv, out, lse, _ = oracle.bwd_frac(q, k, v, g, W, dists)
    rq, rk, rv, ro, rl = oracle.bwd(q, k, v, g, W, S.offset_table(base, Fraction(alpha), W, T))
    for a, b in ((dq, rq), (dk, rk), (dv, rv), (out, ro), (lse, rl)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_bwd_frac_gradient_sums():
    # every query's probabilities sum to 1 and the interpolation weights sum to 1, so
    # sum_j dv_j = sum_i dO_i; sum_k dS_ik = 0 for every query, so sum_j dk_j = 0.
    T, d, W = 300, 8, 5
    q, k, v, g = (rnd((3, T, d), s) for s in (51, 52, 53, 54))
    dists = oracle.frac_distances(f32(0.83), S.FIB, W, T)
    _, dk, dv, _, _, _ = oracle.bwd_frac(q, k, v, g, W, dists)
    np.testing.assert_allclose(dv.sum(axis=1), g.sum(axis=1), rtol=0, atol=1e-10)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, rtol=0, atol=1e-10)
