"""Pins of the oracle's rotary position embedding and the attention through it (CPU only).

Vanilla RoPE: row i, pair (2p, 2p+1) rotated by i * base^(-2p/d). Checked against a
hand-worked rotation, the identity at position 0, norm preservation, the inverse, the
composition of angles, the relative-position property that makes the fixed offsets'
angles in distribution at any length (pt Principais Contribuicoes 3, "Mecanismo"), and
torch autograd through an independent torch statement for the backward.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import schedule as S


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_hand_worked_rotation():
    # d = 4, base 10000: theta = (1, 0.01); row 1 turns pair 0 by 1 rad, pair 1 by 0.01 rad
    x = np.zeros((3, 4))
    x[1] = [1.0, 2.0, 3.0, -1.0]
    x[2] = [0.5, 0.0, 0.0, 1.0]
    y = oracle.rope(x)
    c1, s1, c2, s2 = math.cos(1), math.sin(1), math.cos(0.01), math.sin(0.01)
    np.testing.assert_allclose(y[1], [1 * c1 - 2 * s1, 1 * s1 + 2 * c1,
                                      3 * c2 + 1 * s2, 3 * s2 - 1 * c2], rtol=0, atol=1e-15)
    np.testing.assert_allclose(y[2], [0.5 * math.cos(2), 0.5 * math.sin(2),
                                      -math.sin(0.02), math.cos(0.02)], rtol=0, atol=1e-15)
    np.testing.assert_array_equal(y[0], x[0])


def test_norms_inverse_and_composition():
    x = rnd((2, 3, 50, 16), 1)
    y = oracle.rope(x, base=500.0)
    np.testing.assert_allclose(np.hypot(y[..., 0::2], y[..., 1::2]),
                               np.hypot(x[..., 0::2], x[..., 1::2]), rtol=1e-13, atol=0)
    np.testing.assert_allclose(oracle.rope(y, base=500.0, inverse=True), x, rtol=0, atol=1e-13)
    # rotating row i by i*theta twice = by 2*i*theta: compare with rows 2i of a longer sequence
    z = oracle.rope(oracle.rope(np.ones((50, 16))))
    w = oracle.rope(np.ones((100, 16)))[0::2]
    np.testing.assert_allclose(z, w, rtol=0, atol=1e-12)


def test_scores_depend_only_on_relative_position():
    # shifting both sequences by s rows leaves every rotated score q_i . k_j unchanged
    T, d, s = 40, 32, 13
    q, k = rnd((T, d), 2), rnd((T, d), 3)
    qs, ks = np.zeros((T + s, d)), np.zeros((T + s, d))
    qs[s:], ks[s:] = q, k
    a = oracle.rope(q) @ oracle.rope(k).T
    b = oracle.rope(qs) @ oracle.rope(ks).T
    np.testing.assert_allclose(b[s:, s:], a, rtol=0, atol=1e-11)


def torch_rope(x, base=10000.0):
    T, d = x.shape[-2], x.shape[-1]
    theta = base ** (-2.0 * torch.arange(d // 2, dtype=torch.float64) / d)
    ang = torch.arange(T, dtype=torch.float64)[:, None] * theta[None, :]
    c, s = torch.cos(ang), torch.sin(ang)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    return torch.stack((x0 * c - x1 * s, x0 * s + x1 * c), dim=-1).flatten(-2)


@pytest.mark.parametrize("H,Hkv", [(2, 2), (4, 1)])
def test_rope_attention_matches_torch_and_autograd(H, Hkv):
    B, T, d, W = 1, 120, 16, 6
    tab = S.offset_table(S.FIB, Fraction(1), W, T)
    q, g = rnd((B, H, T, d), 4), rnd((B, H, T, d), 7)
    k, v = rnd((B, Hkv, T, d), 5), rnd((B, Hkv, T, d), 6)
    dq, dk, dv, out, lse = oracle.bwd_rope(q, k, v, g, W, tab)
    o2, _ = oracle.fwd_rope(q, k, v, W, tab)
    np.testing.assert_array_equal(out, o2)
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    m = ((i - j >= 0) & (i - j < W)) | np.isin(i - j, tab)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    G = H // Hkv
    ref = F.scaled_dot_product_attention(torch_rope(tq), torch_rope(tk).repeat_interleave(G, dim=1),
                                         tv.repeat_interleave(G, dim=1),
                                         attn_mask=torch.from_numpy(m), scale=1 / math.sqrt(d))
    (ref * torch.from_numpy(g)).sum().backward()
    np.testing.assert_allclose(out, ref.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-11)
