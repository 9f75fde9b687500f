"""Fractional-offset (learned-alpha) entry points without a GPU: the host tables equal the
oracle's distance lists bit for bit (ceil and weight), integer alphas reproduce the static
tables, and fibattn_fwd_frac rejects bad arguments before touching the device."""
import ctypes
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import static_fibonacci_offset_fibattn_b300 as fa
from oracle import schedule as S


def _alphas():
    g = np.random.default_rng(3)
    xs = list(g.uniform(0.05, 4.0, 40).astype(np.float32)) + [0.5, 1.0, 1.5, 2.0, 3.0, 0.75]
    xs += [np.float32(1.0) - np.float32(2 ** -24), np.float32(1.0) + np.float32(2 ** -23)]
    return [float(np.float32(x)) for x in xs]


@pytest.mark.parametrize("base", [S.FIB, S.POW2])
@pytest.mark.parametrize("WT", [(16, 256), (64, 1024), (1, 64), (6, 4096), (3, 100000)])
def test_frac_tables_match_oracle(base, WT):
    W, T = WT
    for a in _alphas():
        for base_max in (0, 89):
            want = oracle.frac_distances(a, base, W, T, base_max)
            c, w = fa.frac_offsets(a, W, T, base, base_max)
            assert c == [math.ceil(d) for d in want], (a, base_max)
            # the weight is the double ceil(d) - d rounded once to float32
            assert w == [float(np.float32(math.ceil(d) - d)) for d in want], (a, base_max)
            assert all(0.0 <= x < 1.0 for x in w)


@pytest.mark.parametrize("base", [S.FIB, S.POW2])
@pytest.mark.parametrize("WT", [(16, 1 << 30), (1, 100000), (64, 2 ** 31 - 1)])
def test_frac_table_of_a_tiny_alpha_over_an_uncapped_base(base, WT):
    # alpha * F stays below T - 1 for every base value up to 2^63 - 1: the builder visits them
    # all and stops at the cap, without overflowing the next term (it used to loop forever)
    W, T = WT
    a, base_max = float(np.float32(1e-12)), 2 ** 63 - 1
    want = oracle.frac_distances(a, base, W, T, base_max)
    c, w = fa.frac_offsets(a, W, T, base, base_max)
    assert len(want) > 10
    assert c == [math.ceil(d) for d in want]
    assert w == [float(np.float32(math.ceil(d) - d)) for d in want]


@pytest.mark.parametrize("base", [S.FIB, S.POW2])
def test_integer_alpha_gives_static_table(base):
    for a in (1, 2, 3, 5):
        for W, T in ((16, 256), (64, 1024), (2, 5000)):
            c, w = fa.frac_offsets(float(a), W, T, base)
            assert c == S.offset_table(base, Fraction(a), W, T)
            assert w == [0.0] * len(c)


def test_frac_offsets_rejects_bad_arguments():
    for bad in (0.0, -1.0, float("nan"), float("inf"), float(2 ** 21)):
        with pytest.raises(fa.FibAttnError) as e:
            fa.frac_offsets(bad, 16, 256)
        assert e.value.status == fa.INVALID_ARG
    L = fa.lib()
    n = ctypes.c_int32(0)
    assert L.fibattn_frac_offsets(1.0, 7, 0, 16, 256, None, None, 0, ctypes.byref(n)) == fa.INVALID_ARG
    assert L.fibattn_frac_offsets(1.0, 0, -1, 16, 256, None, None, 0, ctypes.byref(n)) == fa.INVALID_ARG
    assert L.fibattn_frac_offsets(1.0, 0, 0, 0, 256, None, None, 0, ctypes.byref(n)) == fa.INVALID_ARG
    # capacity: the needed count is reported
    assert L.fibattn_frac_offsets(1.37, 0, 0, 16, 256, None, None, 0, ctypes.byref(n)) == fa.CAPACITY
    assert n.value == len(oracle.frac_distances(float(np.float32(1.37)), S.FIB, 16, 256))


def _fwd_frac_raw(q=256, B=1, H=1, T=8, d=64, dtype=1, W=4, base=0, base_max=0, alphas=(1.0,),
                  n=None):
    L = fa.lib()
    P = ctypes.c_void_p
    a = None if alphas is None else (ctypes.c_float * max(1, len(alphas)))(*alphas)
    n = len(alphas or ()) if n is None else n
    return L.fibattn_fwd_frac(P(q), P(256), P(256), P(256), P(256), B, H, T, d, dtype, W, 0.0,
                              base, base_max, a, n, None)


def test_fwd_frac_validates_before_launch():
    assert _fwd_frac_raw(q=0) == fa.INVALID_ARG
    assert _fwd_frac_raw(T=(1 << 30) + 1) == fa.INVALID_ARG  # above FIBATTN_T_MAX
    assert _fwd_frac_raw(q=264) == fa.INVALID_ARG          # misaligned
    assert _fwd_frac_raw(alphas=None, n=1) == fa.INVALID_ARG
    assert _fwd_frac_raw(B=0) == fa.INVALID_ARG
    assert _fwd_frac_raw(T=0) == fa.INVALID_ARG
    assert _fwd_frac_raw(W=0) == fa.INVALID_ARG
    assert _fwd_frac_raw(n=0) == fa.INVALID_ARG
    assert _fwd_frac_raw(d=128) == fa.UNSUPPORTED
    assert _fwd_frac_raw(dtype=5) == fa.UNSUPPORTED
    assert _fwd_frac_raw(base=3) == fa.INVALID_ARG
    assert _fwd_frac_raw(alphas=(1.0, 0.0)) == fa.INVALID_ARG  # a bad alpha in any layer
    assert _fwd_frac_raw(alphas=(float("nan"),)) == fa.INVALID_ARG


def test_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fwd_frac(q, q, q, 4, [1.0])
    with pytest.raises(ValueError):
        fa.fwd_frac(q, q, q, 4, [1.0, 2.0])


def _bwd_frac_raw(ptrs=None, dalpha=256, ws=256, ws_bytes=1 << 40, d=64, dtype=1, alphas=(1.3,),
                  base=0):
    L = fa.lib()
    P = ctypes.c_void_p
    ptrs = [256] * 9 if ptrs is None else ptrs
    a = (ctypes.c_float * len(alphas))(*alphas)
    return L.fibattn_bwd_frac(*[P(x) for x in ptrs], P(dalpha), P(ws), ctypes.c_uint64(ws_bytes),
                              1, 1, 8, d, dtype, 4, 0.0, base, 0, a, len(alphas), None)


def test_bwd_frac_validates_before_launch():
    for bad in range(9):
        ptrs = [256] * 9
        ptrs[bad] = 0
        assert _bwd_frac_raw(ptrs) == fa.INVALID_ARG
        ptrs[bad] = 264
        assert _bwd_frac_raw(ptrs) == fa.INVALID_ARG
    assert _bwd_frac_raw(dalpha=0) == fa.INVALID_ARG
    assert _bwd_frac_raw(dalpha=258) == fa.INVALID_ARG
    assert _bwd_frac_raw(ws=0) == fa.INVALID_ARG
    assert _bwd_frac_raw(ws=256 + 16) == fa.INVALID_ARG
    assert _bwd_frac_raw(ws_bytes=16) == fa.INVALID_ARG
    assert _bwd_frac_raw(d=32) == fa.UNSUPPORTED
    assert _bwd_frac_raw(alphas=(1.0, -2.0)) == fa.INVALID_ARG
    assert _bwd_frac_raw(base=5) == fa.INVALID_ARG


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("shape", [(1, 2, 256, 16), (8, 8, 1024, 64), (3, 1, 777, 6)])
def test_bwd_frac_workspace_size_layout(dtype, shape):
    B, H, T, W = shape
    alphas = [0.8, 1.37, 1.9]
    L = fa.lib()
    n = ctypes.c_uint64(0)
    a = (ctypes.c_float * 3)(*alphas)
    assert L.fibattn_bwd_frac_workspace_size(B, H, T, 64, dtype, W, 0, 0, a, 3, ctypes.byref(n)) == fa.OK
    rows = 3 * B * H * T
    a256 = lambda x: (x + 255) // 256 * 256
    if dtype == 0:
        want = a256(rows * 4) + rows * 4
    else:
        n_max = max(len(oracle.frac_distances(f, S.FIB, W, T)) for f in [float(np.float32(x)) for x in alphas])
        rows_pad = 3 * B * H * ((T + 3) // 4 * 4)
        want = a256(2 * a256(rows_pad * 4) + rows_pad * n_max * 4) + rows * 4
    assert n.value == want
