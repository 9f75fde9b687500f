"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, builds host offset tables identical to the oracle's, and rejects bad
arguments with the documented status before touching the device."""
import ctypes
import os
import re
from fractions import Fraction

import pytest
import torch

import static_fibonacci_offset_fibattn_b300 as fa
from oracle import schedule as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"FIBATTN_API\s+[\w\s\*]+?\b(fibattn_\w+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    names = declared_symbols()
    assert len(names) >= 8
    L = fa.lib()
    for n in names:
        assert hasattr(L, n), n
    assert L.fibattn_version() >= 100


def test_status_strings():
    for s in range(6):
        assert fa.status_string(s)
    assert fa.status_string(99) == "unknown status"


def _sched_to_oracle(sc: fa.Schedule, layer, W, T):
    kw = {}
    if sc.kind == "fixed":
        kw["alpha"] = Fraction(*sc.alpha)
    else:
        kw["alpha_min"] = Fraction(*sc.alpha_min)
        kw["alpha_max"] = Fraction(*sc.alpha_max)
        kw["coprime_c"] = sc.coprime_c
    return S.layer_table(sc.base, sc.kind, layer, sc.n_layers, W, T, sc.base_max, **kw)


SCHEDS = [
    fa.Schedule("fixed", "fib", alpha=(1, 1)),
    fa.Schedule("fixed", "pow2", alpha=(1, 1)),
    fa.Schedule("linear", "fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=16),
    fa.Schedule("linear", "fib", alpha_min=(1, 2), alpha_max=(3, 2), n_layers=16),
    fa.Schedule("coprime", "fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=16, coprime_c=5),
    fa.Schedule("coprime", "fib", alpha_min=(1, 2), alpha_max=(3, 2), n_layers=16, coprime_c=7),
    fa.Schedule("linear", "pow2", alpha_min=(1, 2), alpha_max=(3, 2), n_layers=16),
    fa.Schedule("linear", "fib", alpha_min=(3, 2), alpha_max=(1, 3), n_layers=5),
    fa.Schedule("fixed", "fib", alpha=(7, 3), base_max=100000),
    fa.Schedule("fixed", "pow2", alpha=(1, 1000), base_max=0),
    fa.Schedule("coprime", "pow2", alpha_min=(1, 7), alpha_max=(9, 4), n_layers=9, coprime_c=4),
    fa.Schedule("linear", "fib", alpha_min=(5, 4), alpha_max=(5, 4), n_layers=1),
]


@pytest.mark.parametrize("sc", SCHEDS)
@pytest.mark.parametrize("WT", [(16, 256), (64, 1024), (64, 4096), (6, 1024), (12, 100000), (1, 3)])
def test_host_tables_match_oracle(sc, WT):
    W, T = WT
    for layer in range(sc.n_layers):
        want = _sched_to_oracle(sc, layer, W, T)
        if len(want) > fa.MAX_OFFSETS:
            with pytest.raises(fa.FibAttnError) as e:
                fa.offsets(sc, layer, W, T)
            assert e.value.status == fa.CAPACITY
        else:
            assert fa.offsets(sc, layer, W, T) == want, (layer, want)


def test_offsets_rejects_bad_schedules():
    bad = [
        fa.Schedule("coprime", "fib", n_layers=16, coprime_c=4),
        fa.Schedule("coprime", "fib", n_layers=16, coprime_c=0),
        fa.Schedule("fixed", "fib", alpha=(0, 1)),
        fa.Schedule("fixed", "fib", alpha=(1, 0)),
        fa.Schedule("fixed", "fib", alpha=(-1, 2)),
        fa.Schedule("linear", "fib", alpha_min=(1, 2), alpha_max=(1, 0), n_layers=4),
        fa.Schedule("fixed", "fib", alpha=(1 << 21, 1)),
        fa.Schedule("fixed", "fib", n_layers=0),
        fa.Schedule("fixed", "fib", base_max=-1),
    ]
    for sc in bad:
        with pytest.raises(fa.FibAttnError) as e:
            fa.offsets(sc, 0, 16, 256)
        assert e.value.status == fa.INVALID_ARG, sc
    sc = fa.Schedule("fixed", "fib", n_layers=2)
    for (layer, W, T) in [(2, 16, 256), (-1, 16, 256), (0, 0, 256), (0, 16, 0)]:
        with pytest.raises(fa.FibAttnError) as e:
            fa.offsets(sc, layer, W, T)
        assert e.value.status == fa.INVALID_ARG


def test_capacity_status_reports_needed_count():
    L = fa.lib()
    sc = fa.Schedule("fixed", "fib").to_c()
    buf = (ctypes.c_int32 * 2)()
    n = ctypes.c_int32(0)
    st = L.fibattn_offsets(ctypes.byref(sc), 0, 16, 256, buf, 2, ctypes.byref(n))
    assert st == fa.CAPACITY and n.value == 6 and list(buf) == [21, 34]


def _fwd_raw(q=1, k=1, v=1, o=1, lse=1, B=1, H=1, T=8, d=64, dtype=1, W=4, sched=None,
             layer0=0, n=1):
    L = fa.lib()
    sc = (sched or fa.Schedule()).to_c()
    P = lambda x: ctypes.c_void_p(x * 256)  # non-null, 16-byte aligned, never dereferenced
    return L.fibattn_fwd(P(q), P(k), P(v), P(o), P(lse), B, H, T, d, dtype, W, 0.0,
                         ctypes.byref(sc), layer0, n, None)


def test_fwd_validates_before_launch():
    # every one of these is rejected on the host, so no kernel runs (no GPU needed)
    assert _fwd_raw(q=0) == fa.INVALID_ARG
    assert _fwd_raw(B=0) == fa.INVALID_ARG
    assert _fwd_raw(T=0) == fa.INVALID_ARG
    assert _fwd_raw(W=0) == fa.INVALID_ARG
    assert _fwd_raw(d=96) == fa.UNSUPPORTED
    assert _fwd_raw(dtype=7) == fa.UNSUPPORTED
    assert _fwd_raw(n=2) == fa.INVALID_ARG  # schedule has one layer
    assert _fwd_raw(layer0=-1) == fa.INVALID_ARG
    assert _fwd_raw(sched=fa.Schedule("coprime", n_layers=4, coprime_c=2)) == fa.INVALID_ARG
    L = fa.lib()
    sc = fa.Schedule().to_c()
    mis = ctypes.c_void_p(256 + 8)
    ok = ctypes.c_void_p(256)
    assert L.fibattn_fwd(mis, ok, ok, ok, ok, 1, 1, 8, 64, 1, 4, 0.0, ctypes.byref(sc), 0, 1,
                         None) == fa.INVALID_ARG
    assert L.fibattn_fwd(ok, ok, ok, ok, ok, 1, 1, 8, 64, 1, 4, 0.0, None, 0, 1,
                         None) == fa.INVALID_ARG
    # an infinite softmax scale is refused (<= 0 and NaN select 1/sqrt(d))
    assert L.fibattn_fwd(ok, ok, ok, ok, ok, 1, 1, 8, 64, 1, 4, float("inf"), ctypes.byref(sc),
                         0, 1, None) == fa.INVALID_ARG


def _header_define(name):
    text = open(os.path.join(ROOT, "include", "fibattn.h")).read()
    m = re.search(r"#define\s+" + name + r"\s+\(1 << (\d+)\)", text)
    return 1 << int(m.group(1))


def test_sequence_length_limit():
    # T above FIBATTN_T_MAX is rejected on the host by every call that launches work (tile
    # and padded row counts of T + 127 or T + 31 would leave 32 bits); the host table call
    # still takes any T
    TM = _header_define("FIBATTN_T_MAX")
    assert TM == 1 << 30
    L = fa.lib()
    sc = fa.Schedule().to_c()
    ok = ctypes.c_void_p(256)
    for T in (TM + 1, 2 ** 31 - 1):
        assert _fwd_raw(T=T) == fa.INVALID_ARG
        n = ctypes.c_uint64(0)
        assert L.fibattn_bwd_workspace_size(1, 1, T, 64, 1, 4, ctypes.byref(sc), 0, 1,
                                            ctypes.byref(n)) == fa.INVALID_ARG
        assert L.fibattn_keyset_debug(ctypes.byref(sc), 0, 4, T, ok, None) == fa.INVALID_ARG
        assert L.fibattn_offsets_device(ctypes.byref(sc), 0, 1, 4, T, ok, ok, None) == fa.INVALID_ARG
        assert L.fibattn_rope_table(ok, T, 64, ctypes.c_double(1e4), None) == fa.INVALID_ARG
        assert L.fibattn_rope(ok, ok, 1, T, 64, 1, ok, T, 0, None) == fa.INVALID_ARG
    buf = (ctypes.c_int32 * 64)()
    cnt = ctypes.c_int32(0)
    assert L.fibattn_offsets(ctypes.byref(sc), 0, 4, 2 ** 31 - 1, buf, 64, ctypes.byref(cnt)) == fa.OK
    assert list(buf[: cnt.value]) == S.offset_table(S.FIB, Fraction(1), 4, 2 ** 31 - 1)


def test_bwd_validates_before_launch():
    L = fa.lib()
    sc = fa.Schedule().to_c()
    ok = ctypes.c_void_p(256)
    big = ctypes.c_uint64(1 << 40)
    args = [ok] * 10
    for bad in range(10):
        a = list(args)
        a[bad] = ctypes.c_void_p(0)
        assert L.fibattn_bwd(*a, big, 1, 1, 8, 64, 1, 4, 0.0, ctypes.byref(sc), 0, 1,
                             None) == fa.INVALID_ARG
    assert L.fibattn_bwd(*args, big, 1, 1, 8, 32, 1, 4, 0.0, ctypes.byref(sc), 0, 1,
                         None) == fa.UNSUPPORTED
    # a workspace that is not 256-byte aligned, or too small, is rejected before any launch
    a = list(args)
    a[9] = ctypes.c_void_p(256 + 16)
    assert L.fibattn_bwd(*a, big, 1, 1, 8, 64, 1, 4, 0.0, ctypes.byref(sc), 0, 1,
                         None) == fa.INVALID_ARG
    assert L.fibattn_bwd(*args, ctypes.c_uint64(16), 1, 1, 8, 64, 1, 4, 0.0, ctypes.byref(sc),
                         0, 1, None) == fa.INVALID_ARG


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("shape", [(1, 2, 256, 16), (8, 8, 1024, 64), (2, 8, 4096, 64),
                                   (3, 1, 777, 6)])
def test_bwd_workspace_size_layout(dtype, shape):
    # f32: D (4 bytes per row). bf16: rows padded to a multiple of 4; D and lse*log2(e)
    # (4 bytes per padded row each, each array 256-aligned) and one 4-byte (P, dS) pair per
    # padded row and table slot, n_max = the largest of the call's tables (from the oracle)
    B, H, T, W = shape
    sched = dict(kind="coprime", base="fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=16,
                 coprime_c=5)
    sc = fa.Schedule(**sched).to_c()
    n = ctypes.c_uint64(0)
    a256 = lambda x: (x + 255) // 256 * 256
    for layer0, Lc in ((0, 16), (3, 5), (15, 1)):
        assert fa.lib().fibattn_bwd_workspace_size(B, H, T, 64, dtype, W, ctypes.byref(sc),
                                                   layer0, Lc, ctypes.byref(n)) == fa.OK
        sc_py = fa.Schedule(**sched)
        n_max = max(len(_sched_to_oracle(sc_py, l, W, T)) for l in range(layer0, layer0 + Lc))
        if dtype == 0:
            want = Lc * B * H * T * 4
        else:
            rows = Lc * B * H * ((T + 3) // 4 * 4)
            want = 2 * a256(rows * 4) + rows * n_max * 4
        assert n.value == want


def test_binding_refuses_cpu_tensors():
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fwd(q, q, q, 4, fa.Schedule())


def test_bwd_noalloc_rejects_oversize_on_the_host():
    # a call whose workspace exceeds the fixed array: SCRATCH_LIMIT, decided before any
    # CUDA call. 16 layers x B=16 x H=8 x T=1024 needs 4 + 4 + 4 * 6 bytes per row = 64 MiB.
    L = fa.lib()
    sc = fa.Schedule("coprime", "fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=16,
                     coprime_c=5).to_c()
    ok = ctypes.c_void_p(256)
    n = ctypes.c_uint64(0)
    assert L.fibattn_bwd_workspace_size(16, 8, 1024, 64, 1, 64, ctypes.byref(sc), 0, 16,
                                        ctypes.byref(n)) == fa.OK
    assert n.value > fa.NOALLOC_SCRATCH_BYTES
    st = L.fibattn_bwd_noalloc(*([ok] * 9), 16, 8, 1024, 64, 1, 64, 0.0, ctypes.byref(sc), 0, 16,
                               None)
    assert st == fa.SCRATCH_LIMIT
    assert "scratch" in fa.status_string(fa.SCRATCH_LIMIT)
    # the 16-layer B=8 training-step shape fits (32 MiB)
    assert L.fibattn_bwd_workspace_size(8, 8, 1024, 64, 1, 64, ctypes.byref(sc), 0, 16,
                                        ctypes.byref(n)) == fa.OK
    assert n.value <= fa.NOALLOC_SCRATCH_BYTES


def test_gqa_entry_points_validate_before_launch():
    L = fa.lib()
    sc = fa.Schedule().to_c()
    ok = ctypes.c_void_p(256)
    big = ctypes.c_uint64(1 << 40)
    for H, Hkv in ((6, 4), (4, 0), (4, -1), (0, 1)):
        assert L.fibattn_fwd_gqa(ok, ok, ok, ok, ok, 1, H, Hkv, 8, 64, 1, 4, 0.0, ctypes.byref(sc),
                                 0, 1, None) == fa.INVALID_ARG
        assert L.fibattn_bwd_gqa(*([ok] * 10), big, 1, H, Hkv, 8, 64, 1, 4, 0.0, ctypes.byref(sc),
                                 0, 1, None) == fa.INVALID_ARG
    assert L.fibattn_fwd_gqa(ok, ok, ok, ok, ok, 1, 4, 2, 8, 32, 1, 4, 0.0, ctypes.byref(sc), 0, 1,
                             None) == fa.UNSUPPORTED


def test_binding_checks_kv_head_shapes():
    q = torch.zeros(1, 6, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fwd(q, torch.zeros(1, 4, 8, 64, dtype=torch.bfloat16),
               torch.zeros(1, 4, 8, 64, dtype=torch.bfloat16), 4, fa.Schedule())
    with pytest.raises(ValueError):
        fa.fwd(q, torch.zeros(1, 3, 8, 64, dtype=torch.bfloat16),
               torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16), 4, fa.Schedule())


def test_outputs_must_not_overlap_inputs():
    # every argument is valid except that an output shares bytes with an input or another
    # output, so the overlap check is what rejects these calls, before any launch
    L = fa.lib()
    sc = fa.Schedule().to_c()
    P = lambda mib, off=0: ctypes.c_void_p((mib << 20) + off)  # 1 MiB apart: disjoint here
    B, H, T, d, W = 1, 1, 8, 64, 4                              # 1 KB per bf16 tensor
    fwd = lambda q, k, v, o, lse: L.fibattn_fwd(q, k, v, o, lse, B, H, T, d, 1, W, 0.0,
                                                 ctypes.byref(sc), 0, 1, None)
    assert fwd(P(1), P(2), P(3), P(1), P(5)) == fa.INVALID_ARG          # o is q
    assert fwd(P(1), P(2), P(3), P(4), P(4, 512)) == fa.INVALID_ARG     # lse inside o
    assert fwd(P(1), P(2), P(3), P(3, 1008), P(5)) == fa.INVALID_ARG    # o's start in v
    need = ctypes.c_uint64(0)
    assert L.fibattn_bwd_workspace_size(B, H, T, d, 1, W, ctypes.byref(sc), 0, 1,
                                        ctypes.byref(need)) == fa.OK
    ws = ctypes.c_uint64(need.value)

    def bwd(dq, dk, dv, wsp):
        return L.fibattn_bwd(P(1), P(2), P(3), P(4), P(5), P(6), dq, dk, dv, wsp, ws, B, H, T, d,
                             1, W, 0.0, ctypes.byref(sc), 0, 1, None)

    assert bwd(P(7), P(2), P(9), P(10)) == fa.INVALID_ARG    # dk is k
    assert bwd(P(7), P(8), P(8), P(10)) == fa.INVALID_ARG    # dk is dv
    assert bwd(P(7), P(8), P(9), P(7)) == fa.INVALID_ARG     # the workspace over dq
    assert bwd(P(6), P(8), P(9), P(10)) == fa.INVALID_ARG    # dq over dO


def test_binding_checks_lse():
    # a caller-given lse must be float32, shaped q.shape[:-1], contiguous, on q's device:
    # otherwise the forward would write (or the backward read) past its end
    q = torch.empty(2, 3, 8, 64)
    fa._check_lse(torch.empty(2, 3, 8), q)
    for bad in (torch.empty(2, 3, 8, dtype=torch.bfloat16), torch.empty(2, 3, 7),
                torch.empty(2, 3, 16)[:, :, ::2], torch.empty(6, 8), torch.empty(2, 3, 8, 1)):
        with pytest.raises(ValueError):
            fa._check_lse(bad, q)


def test_rope_entry_points_validate_before_launch():
    L = fa.lib()
    sc = fa.Schedule().to_c()
    ok = ctypes.c_void_p(256)
    assert L.fibattn_rope_table(ok, 8, 64, ctypes.c_double(1.0), None) == fa.INVALID_ARG
    assert L.fibattn_rope_table(ok, 0, 64, ctypes.c_double(1e4), None) == fa.INVALID_ARG
    assert L.fibattn_rope_table(ok, 8, 32, ctypes.c_double(1e4), None) == fa.UNSUPPORTED
    # table shorter than T, partial overlap, misalignment
    assert L.fibattn_rope(ok, ok, 1, 8, 64, 1, ok, 4, 0, None) == fa.INVALID_ARG
    assert L.fibattn_rope(ok, ctypes.c_void_p(256 + 128), 1, 8, 64, 1, ok, 8, 0, None) == fa.INVALID_ARG
    assert L.fibattn_rope(ctypes.c_void_p(264), ok, 1, 8, 64, 1, ok, 8, 0, None) == fa.INVALID_ARG
    assert L.fibattn_rope(ok, ok, 1, 8, 64, 3, ok, 8, 0, None) == fa.UNSUPPORTED
    # more than 2^40 rows, also where slices * T would wrap around in 64 bits
    assert L.fibattn_rope(ok, ok, (1 << 38) + 1, 4, 64, 1, ok, 8, 0, None) == fa.INVALID_ARG
    assert L.fibattn_rope(ok, ok, (1 << 62) + 1, 4, 64, 1, ok, 8, 0, None) == fa.INVALID_ARG
    assert L.fibattn_fwd_rope(*([ok] * 7), 1, 4, 2, 8, 64, 1, 4, 0.0, ctypes.byref(sc), 0, 1, ok, 7,
                              None) == fa.INVALID_ARG
    assert L.fibattn_fwd_rope(*([ok] * 7), 1, 4, 3, 8, 64, 1, 4, 0.0, ctypes.byref(sc), 0, 1, ok, 8,
                              None) == fa.INVALID_ARG
    assert L.fibattn_bwd_rope(*([ok] * 10), ctypes.c_uint64(1 << 40), 1, 4, 2, 8, 64, 1, 4, 0.0,
                              ctypes.byref(sc), 0, 1, None, 8, None) == fa.INVALID_ARG
    # the fused form: a short table, bad head counts, then fp32 and head size 128 unsupported
    fused = L.fibattn_fwd_rope_fused
    assert fused(*([ok] * 5), 1, 4, 2, 8, 64, 1, 4, 0.0, ctypes.byref(sc), 0, 1, ok, 7,
                 None) == fa.INVALID_ARG
    assert fused(*([ok] * 5), 1, 4, 3, 8, 64, 1, 4, 0.0, ctypes.byref(sc), 0, 1, ok, 8,
                 None) == fa.INVALID_ARG
    assert fused(*([ok] * 5), 1, 4, 2, 8, 64, 0, 4, 0.0, ctypes.byref(sc), 0, 1, ok, 8,
                 None) == fa.UNSUPPORTED
    assert fused(*([ok] * 5), 1, 4, 2, 8, 128, 1, 4, 0.0, ctypes.byref(sc), 0, 1, ok, 8,
                 None) == fa.UNSUPPORTED


def test_debug_wait_timeout_validates_before_launch():
    L = fa.lib()
    for bad in (0, -5, 10001):
        assert L.fibattn_debug_wait_timeout(bad, None) == fa.INVALID_ARG


def test_bwd_fused_validates_before_launch():
    # null or misaligned pointers, a misaligned or short workspace: INVALID_ARG; fp32, head
    # size 128 or a bad head size: UNSUPPORTED; all decided on the host before any launch
    L = fa.lib()
    sc = fa.Schedule().to_c()
    ok = ctypes.c_void_p(256)
    big = ctypes.c_uint64(1 << 40)
    args = [ok] * 10
    tail = (1, 1, 8, 64, 1, 4, 0.0, ctypes.byref(sc), 0, 1, None)
    for bad in range(10):
        a = list(args)
        a[bad] = ctypes.c_void_p(0)
        assert L.fibattn_bwd_fused(*a, big, *tail) == fa.INVALID_ARG
    a = list(args)
    a[0] = ctypes.c_void_p(256 + 8)
    assert L.fibattn_bwd_fused(*a, big, *tail) == fa.INVALID_ARG
    a = list(args)
    a[9] = ctypes.c_void_p(256 + 16)
    assert L.fibattn_bwd_fused(*a, big, *tail) == fa.INVALID_ARG
    # B1 H1 T8: two 256-aligned arrays of 8 floats = 512 bytes
    assert L.fibattn_bwd_fused(*args, ctypes.c_uint64(511), *tail) == fa.INVALID_ARG
    for d, dtype in ((64, 0), (128, 1), (32, 1)):
        assert L.fibattn_bwd_fused(*args, big, 1, 1, 8, d, dtype, 4, 0.0, ctypes.byref(sc), 0, 1,
                                   None) == fa.UNSUPPORTED


def test_bwd_fused_workspace_size_is_d_and_lse_only():
    q = torch.empty(16, 8, 8, 1023, 64, dtype=torch.bfloat16, device="meta")
    rows = 16 * 8 * 8 * 1024
    assert fa.bwd_fused_workspace_size(q) == 2 * ((rows * 4 + 255) // 256 * 256)


def test_fwd_bwd_validates_before_launch():
    # null or misaligned pointers, n_streams out of [1, 8], a misaligned or short workspace:
    # INVALID_ARG; a bad head size: UNSUPPORTED; all decided on the host before any launch
    L = fa.lib()
    sc = fa.Schedule().to_c()
    ok = ctypes.c_void_p(256)
    big = ctypes.c_uint64(1 << 40)
    args = [ok] * 10
    tail = lambda ns, d=64: (1, 1, 1, 8, d, 1, 4, 0.0, ctypes.byref(sc), 0, 1, ns, None)
    for bad in range(10):
        a = list(args)
        a[bad] = ctypes.c_void_p(0)
        assert L.fibattn_fwd_bwd(*a, big, *tail(2)) == fa.INVALID_ARG
    for ns in (0, 9, -1):
        assert L.fibattn_fwd_bwd(*args, big, *tail(ns)) == fa.INVALID_ARG
    a = list(args)
    a[9] = ctypes.c_void_p(256 + 16)
    assert L.fibattn_fwd_bwd(*a, big, *tail(2)) == fa.INVALID_ARG
    assert L.fibattn_fwd_bwd(*args, ctypes.c_uint64(16), *tail(2)) == fa.INVALID_ARG
    assert L.fibattn_fwd_bwd(*args, big, *tail(2, d=32)) == fa.UNSUPPORTED


@pytest.mark.parametrize("n_streams", [1, 2, 3, 8])
def test_fwd_bwd_workspace_is_the_groups_workspaces(n_streams):
    # the layers split into min(n_streams, Lc) contiguous groups; the workspace is each group's
    # backward workspace, 256-aligned, one after the other
    sched = dict(kind="coprime", base="fib", alpha_min=(1, 2), alpha_max=(2, 1), n_layers=16,
                 coprime_c=5)
    sc = fa.Schedule(**sched).to_c()
    L = fa.lib()
    B, H, T, W, layer0, Lc = 2, 8, 1000, 64, 1, 13
    got = ctypes.c_uint64(0)
    assert L.fibattn_fwd_bwd_workspace_size(B, H, T, 64, 1, W, ctypes.byref(sc), layer0, Lc,
                                            n_streams, ctypes.byref(got)) == fa.OK
    groups = min(n_streams, Lc)
    want = 0
    for g in range(groups):
        a, b = Lc * g // groups, Lc * (g + 1) // groups
        n = ctypes.c_uint64(0)
        assert L.fibattn_bwd_workspace_size(B, H, T, 64, 1, W, ctypes.byref(sc), layer0 + a, b - a,
                                            ctypes.byref(n)) == fa.OK
        want += (n.value + 255) // 256 * 256
    assert got.value == want
