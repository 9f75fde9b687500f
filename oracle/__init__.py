"""The oracle: slow, obviously correct CPU statement of Fibonacci-offset sparse attention.

TEST INFRASTRUCTURE ONLY. Only `tests/`, `__graft_entry__.smoke()` and the
benchmark's CPU-baseline / reference leg may import this package. The CUDA
library never calls it, and the two share no code: this package computes offsets
with Python `fractions.Fraction` (schedule.py) and attention in a separate fp64
C file (fibattn_oracle.c), loaded here through ctypes.

Source: "Depth-Staggered Fibonacci Spacing for Sparse Attention: Static Schedules
Beat Learned Dilation and Extrapolate Where Dense Attention Fails" (gist.science
explainer, Metodologia; aimsg.uk summary, core content). See schedule.py and
fibattn_oracle.c for the step-by-step citations.

Parity pins (tests/test_oracle_*.py): the printed Fibonacci list and Binet's
formula, the schedule endpoints and the coprime multiset, the power-of-two
offsets the pages name at 4x length, dense causal attention (W >= T), sliding
window attention (empty table), the library masked-attention routine with a
brute-force mask, V = 1, Q = 0, the first query, and central finite differences
plus autograd for the backward; for fractional offsets, the integer-alpha reduction,
values linear in position, keys linear in position (closed-form scores), and
continuity at integer alpha.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

from . import schedule
from .schedule import (FIB, POW2, FIXED, LINEAR, COPRIME, alpha_for_layer, fibonacci_base,
                       frac_bases, frac_distances, key_set, layer_table, offset_table,
                       round_half_up)

_lib = None


def lib():
    global _lib
    if _lib is None:
        from .build import build
        path = build()
        L = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        i64 = ctypes.c_int64
        L.oracle_fwd.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i64, ctypes.c_double,
                                 ip, ip, i64, ip, ctypes.c_int]
        L.oracle_fwd.restype = ctypes.c_int
        L.oracle_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp, i64, i64, i64, i64,
                                 ctypes.c_double, ip, ip, i64, ip, ctypes.c_int]
        L.oracle_bwd.restype = ctypes.c_int
        L.oracle_key_set.argtypes = [i64, i64, ip, ctypes.c_int, ctypes.POINTER(ctypes.c_int64)]
        L.oracle_key_set.restype = i64
        L.oracle_fwd_frac.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i64, ctypes.c_double,
                                      dp, ip, i64, ip, ctypes.c_int]
        L.oracle_fwd_frac.restype = ctypes.c_int
        L.oracle_bwd_frac.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, i64, i64, i64, i64,
                                      ctypes.c_double, dp, ip, i64, ip, ctypes.c_int]
        L.oracle_bwd_frac.restype = ctypes.c_int
        L.oracle_threads.argtypes = [ctypes.c_int]
        L.oracle_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _dptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _iptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _pack_tables(tables):
    cap = max([1] + [len(t) for t in tables])
    arr = np.zeros((len(tables), cap), dtype=np.int32)
    cnt = np.zeros(len(tables), dtype=np.int32)
    for r, t in enumerate(tables):
        arr[r, :len(t)] = t
        cnt[r] = len(t)
    return arr, cnt, cap


def _as_slices(x):
    x = np.ascontiguousarray(x, dtype=np.float64)
    T, d = x.shape[-2], x.shape[-1]
    return x.reshape(-1, T, d), x.shape


def threads(n: int = 0) -> int:
    """Threads the oracle's OpenMP loop uses (n > 0 sets it)."""
    return lib().oracle_threads(int(n))


def key_set_c(i: int, W: int, table):
    """The C oracle's materialised key set of query i (cross-checked against schedule.key_set)."""
    tab = np.asarray(table, dtype=np.int32)
    out = np.zeros(i + len(tab) + 2, dtype=np.int64)
    n = lib().oracle_key_set(int(i), int(W), _iptr(tab), len(tab),
                             out.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)))
    return out[:n].tolist()


def _slice_tables(shape, tables):
    """tables: one table per index of the leading axis (a layer each), or one flat
    table for every slice. Returns the table list and each slice's table index."""
    n_slices = int(np.prod(shape[:-2], dtype=np.int64))
    per_layer_tables = len(tables) > 0 and isinstance(tables[0], (list, tuple, np.ndarray))
    if per_layer_tables:
        if len(shape) < 3 or len(tables) != shape[0]:
            raise ValueError("need one table per index of the leading axis")
        tabs = [[int(o) for o in t] for t in tables]
        per = n_slices // shape[0]
    else:
        tabs = [[int(o) for o in tables]]
        per = n_slices
    tos = np.repeat(np.arange(len(tabs), dtype=np.int32), per)
    return tabs, tos


def fwd(q, k, v, W: int, tables, scale: float | None = None, n_threads: int = 0):
    """Sparse attention forward in fp64.

    q, k, v: arrays [..., T, d] (any leading dims; with a table per leading index when
    `tables` is a list of lists, else one table for all). Returns (out, lse)."""
    qs, shape = _as_slices(q)
    ks, _ = _as_slices(k)
    vs, _ = _as_slices(v)
    T, d = shape[-2], shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    tabs, tos = _slice_tables(shape, tables)
    arr, cnt, cap = _pack_tables(tabs)
    out = np.zeros_like(qs)
    lse = np.zeros(qs.shape[:-1], dtype=np.float64)
    rc = lib().oracle_fwd(_dptr(qs), _dptr(ks), _dptr(vs), _dptr(out), _dptr(lse), qs.shape[0], T,
                          d, int(W), float(scale), _iptr(arr), _iptr(cnt), cap, _iptr(tos),
                          int(n_threads))
    if rc:
        raise MemoryError("oracle_fwd failed")
    return out.reshape(shape), lse.reshape(shape[:-1])


def _repeat_kv(x, G: int):
    """Grouped-query layout: [..., H_kv, T, d] -> [..., H_kv * G, T, d], query head h reading
    kv head h // G (consecutive query heads share one kv head)."""
    return np.repeat(np.asarray(x, dtype=np.float64), G, axis=-3)


def fwd_gqa(q, k, v, W: int, tables, scale: float | None = None, n_threads: int = 0):
    """Forward with grouped K/V heads: q [..., H, T, d], k and v [..., H_kv, T, d] with
    H = G * H_kv. By the definition of sharing, every query head attends its kv head's rows:
    the multi-head forward over the repeated K/V."""
    G = _group(q, k)
    return fwd(q, _repeat_kv(k, G), _repeat_kv(v, G), W, tables, scale, n_threads)


def bwd_gqa(q, k, v, dout, W: int, tables, scale: float | None = None, n_threads: int = 0):
    """Backward with grouped K/V heads: a shared kv row's gradient is the sum of the gradients
    of its G copies. Returns (dq, dk, dv, out, lse) with dk, dv shaped like k, v."""
    G = _group(q, k)
    dq, dk, dv, out, lse = bwd(q, _repeat_kv(k, G), _repeat_kv(v, G), dout, W, tables, scale,
                               n_threads)
    shp = np.shape(k)
    red = lambda a: a.reshape(shp[:-3] + (shp[-3], G) + shp[-2:]).sum(axis=-3)
    return dq, red(dk), red(dv), out, lse


def _group(q, k):
    H, Hkv = np.shape(q)[-3], np.shape(k)[-3]
    if Hkv < 1 or H % Hkv or np.shape(q)[:-3] != np.shape(k)[:-3]:
        raise ValueError("q heads must be a multiple of the kv heads, other dims equal")
    return H // Hkv


def rope(x, base: float = 10000.0, inverse: bool = False):
    """Vanilla rotary position embedding in fp64 (pt Significancia: the models use RoPE
    without scaling; Metodologia / Arquitetura, "Implementacao": RoPE is applied before the
    gather). Row i of every [..., T, d] slice has each pair (2p, 2p+1) rotated by the angle
    i * theta_p, theta_p = base^(-2p/d); `inverse` rotates by the opposite angle (the
    transpose, which carries gradients back through the rotation)."""
    x = np.asarray(x, dtype=np.float64)
    T, d = x.shape[-2], x.shape[-1]
    if d % 2:
        raise ValueError("d must be even")
    theta = float(base) ** (-2.0 * np.arange(d // 2, dtype=np.float64) / d)
    ang = np.arange(T, dtype=np.float64)[:, None] * theta[None, :]
    c, s = np.cos(ang), np.sin(ang)
    if inverse:
        s = -s
    x0, x1 = x[..., 0::2], x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = x0 * c - x1 * s
    y[..., 1::2] = x0 * s + x1 * c
    return y


def fwd_rope(q, k, v, W: int, tables, base: float = 10000.0, scale: float | None = None,
             n_threads: int = 0):
    """Forward with RoPE applied to q and k before the attention (kv heads may be grouped)."""
    return fwd_gqa(rope(q, base), rope(k, base), v, W, tables, scale, n_threads)


def bwd_rope(q, k, v, dout, W: int, tables, base: float = 10000.0, scale: float | None = None,
             n_threads: int = 0):
    """Backward through RoPE: the attention gradients of the rotated q and k, rotated back."""
    dq, dk, dv, out, lse = bwd_gqa(rope(q, base), rope(k, base), v, dout, W, tables, scale,
                                   n_threads)
    return rope(dq, base, inverse=True), rope(dk, base, inverse=True), dv, out, lse


def _frac_tables(dist_tables, shape, n_slices):
    per_layer = len(dist_tables) > 0 and isinstance(dist_tables[0], (list, tuple, np.ndarray))
    tabs = [list(map(float, t)) for t in dist_tables] if per_layer else [list(map(float, dist_tables))]
    if per_layer and (len(shape) < 3 or len(tabs) != shape[0]):
        raise ValueError("need one distance list per index of the leading axis")
    tos = np.repeat(np.arange(len(tabs), dtype=np.int32), n_slices // len(tabs))
    cap = max([1] + [len(t) for t in tabs])
    arr = np.zeros((len(tabs), cap), dtype=np.float64)
    cnt = np.zeros(len(tabs), dtype=np.int32)
    for r, t in enumerate(tabs):
        arr[r, :len(t)] = t
        cnt[r] = len(t)
    return arr, cnt, cap, tos


def fwd_frac(q, k, v, W: int, dist_tables, scale: float | None = None, n_threads: int = 0):
    """Forward with fractional offsets in fp64: dist_tables is one list of real distances
    (schedule.frac_distances) per index of the leading axis, or one list for all slices.
    Returns (out, lse)."""
    qs, shape = _as_slices(q)
    ks, _ = _as_slices(k)
    vs, _ = _as_slices(v)
    T, d = shape[-2], shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    n_slices = qs.shape[0]
    arr, cnt, cap, tos = _frac_tables(dist_tables, shape, n_slices)
    out = np.zeros_like(qs)
    lse = np.zeros(qs.shape[:-1], dtype=np.float64)
    rc = lib().oracle_fwd_frac(_dptr(qs), _dptr(ks), _dptr(vs), _dptr(out), _dptr(lse), n_slices,
                               T, d, int(W), float(scale), _dptr(arr), _iptr(cnt), cap,
                               _iptr(tos), int(n_threads))
    if rc:
        raise MemoryError("oracle_fwd_frac failed")
    return out.reshape(shape), lse.reshape(shape[:-1])


def bwd_frac(q, k, v, dout, W: int, dist_tables, scale: float | None = None, n_threads: int = 0):
    """Backward with fractional offsets in fp64 (tables as in fwd_frac). Returns
    (dq, dk, dv, out, lse, dd) where dd[..., t] = dL/dd_t of each slice for the loss
    L = sum(dout * out); dL/dalpha of a layer is sum over its slices of sum_t f_t dd[..., t]."""
    qs, shape = _as_slices(q)
    ks, _ = _as_slices(k)
    vs, _ = _as_slices(v)
    gs, _ = _as_slices(dout)
    T, d = shape[-2], shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    n_slices = qs.shape[0]
    arr, cnt, cap, tos = _frac_tables(dist_tables, shape, n_slices)
    dq, dk, dv, out = (np.zeros_like(qs) for _ in range(4))
    lse = np.zeros(qs.shape[:-1], dtype=np.float64)
    dd = np.zeros((n_slices, cap), dtype=np.float64)
    rc = lib().oracle_bwd_frac(_dptr(qs), _dptr(ks), _dptr(vs), _dptr(gs), _dptr(dq), _dptr(dk),
                               _dptr(dv), _dptr(out), _dptr(lse), _dptr(dd), n_slices, T, d,
                               int(W), float(scale), _dptr(arr), _iptr(cnt), cap, _iptr(tos),
                               int(n_threads))
    if rc:
        raise MemoryError("oracle_bwd_frac failed")
    r = lambda a: a.reshape(shape)
    return (r(dq), r(dk), r(dv), r(out), lse.reshape(shape[:-1]),
            dd.reshape(tuple(shape[:-2]) + (cap,)))


def bwd(q, k, v, dout, W: int, tables, scale: float | None = None, n_threads: int = 0):
    """Sparse attention backward in fp64. Returns (dq, dk, dv, out, lse)."""
    qs, shape = _as_slices(q)
    ks, _ = _as_slices(k)
    vs, _ = _as_slices(v)
    gs, _ = _as_slices(dout)
    T, d = shape[-2], shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    tabs, tos = _slice_tables(shape, tables)
    arr, cnt, cap = _pack_tables(tabs)
    out = np.zeros_like(qs)
    lse = np.zeros(qs.shape[:-1], dtype=np.float64)
    dq = np.zeros_like(qs)
    dk = np.zeros_like(qs)
    dv = np.zeros_like(qs)
    rc = lib().oracle_bwd(_dptr(qs), _dptr(ks), _dptr(vs), _dptr(gs), _dptr(out), _dptr(lse),
                          _dptr(dq), _dptr(dk), _dptr(dv), qs.shape[0], T, d, int(W),
                          float(scale), _iptr(arr), _iptr(cnt), cap, _iptr(tos), int(n_threads))
    if rc:
        raise MemoryError("oracle_bwd failed")
    r = lambda a: a.reshape(shape)
    return r(dq), r(dk), r(dv), r(out), lse.reshape(shape[:-1])


__all__ = ["schedule", "FIB", "POW2", "FIXED", "LINEAR", "COPRIME", "alpha_for_layer",
           "fibonacci_base", "frac_distances", "key_set", "key_set_c", "layer_table",
           "offset_table", "round_half_up", "fwd", "fwd_frac", "bwd", "bwd_frac", "frac_bases",
           "fwd_gqa", "bwd_gqa", "rope", "fwd_rope", "bwd_rope",
           "threads", "lib"]
