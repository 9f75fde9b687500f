"""Python binding of libfibattn (B300 / sm_103a Fibonacci-offset sparse attention).

Argument marshalling only: every step of the computation runs in the CUDA kernels
behind the C ABI declared in include/fibattn.h. PyTorch provides device memory and
the current stream. There is no CPU fallback: if the library is missing or the
tensors are not on a CUDA device, these functions raise.

Attention computed ("Depth-Staggered Fibonacci Spacing for Sparse Attention",
gist.science explainer, Metodologia / Arquitetura e Mecanismo de Atencao): query i
of layer l attends the window i-W+1..i plus i - o for every o in the layer's
offset table, o = round(alpha_l * F) over the Fibonacci (or power-of-two) base.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass, field
from typing import Optional, Sequence, Tuple

import torch

__all__ = ["Schedule", "FibAttnError", "offsets", "offsets_device", "fwd", "bwd",
           "keyset_debug", "poll_device_error", "status_string", "lib", "library_path",
           "FibSparseAttention", "MAX_OFFSETS", "bwd_noalloc", "NOALLOC_SCRATCH_BYTES",
           "bwd_workspace_size", "last_cuda_error", "frac_offsets", "fwd_frac", "bwd_frac",
           "bwd_frac_workspace_size", "FibFracAttention", "rope_table", "rope", "fwd_rope",
           "bwd_rope", "fwd_rope_fused", "bwd_fused", "bwd_fused_workspace_size",
           "fwd_bwd", "fwd_bwd_workspace_size", "STEP_STREAMS_MAX", "debug_wait_timeout"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libfibattn.so")
MAX_OFFSETS = 64

OK, INVALID_ARG, UNSUPPORTED, CAPACITY, CUDA_ERR, TIMEOUT, SCRATCH_LIMIT = range(7)
NOALLOC_SCRATCH_BYTES = 40 << 20
STEP_STREAMS_MAX = 8
_BASES = {"fib": 0, "pow2": 1}
_KINDS = {"fixed": 0, "linear": 1, "coprime": 2}
_DTYPES = {torch.float32: 0, torch.bfloat16: 1}


class FibAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = f"{where}: {status_string(status)} (status {status})"
        self.cuda_error = None
        if status == CUDA_ERR:
            self.cuda_error, call = last_cuda_error()
            msg += f"; CUDA error {self.cuda_error} in {call}"
        super().__init__(msg)
        self.status = status


class _Ratio(ctypes.Structure):
    _fields_ = [("num", ctypes.c_int32), ("den", ctypes.c_int32)]


class _Sched(ctypes.Structure):
    _fields_ = [("base", ctypes.c_int32), ("kind", ctypes.c_int32), ("alpha", _Ratio),
                ("alpha_min", _Ratio), ("alpha_max", _Ratio), ("n_layers", ctypes.c_int32),
                ("coprime_c", ctypes.c_int32), ("base_max", ctypes.c_int64)]


@dataclass(frozen=True)
class Schedule:
    """A per-layer alpha schedule; ratios are (numerator, denominator) pairs.

    kind: 'fixed' (alpha everywhere), 'linear' (alpha_min -> alpha_max across
    n_layers), 'coprime' (the linear alphas reassigned l -> coprime_c*l mod n_layers).
    base: 'fib' (1, 2, 3, ..., 987) or 'pow2' (powers of two)."""
    kind: str = "fixed"
    base: str = "fib"
    alpha: Tuple[int, int] = (1, 1)
    alpha_min: Tuple[int, int] = (1, 2)
    alpha_max: Tuple[int, int] = (3, 2)
    n_layers: int = 1
    coprime_c: int = 7
    base_max: int = 0

    def to_c(self) -> _Sched:
        return _Sched(_BASES[self.base], _KINDS[self.kind], _Ratio(*self.alpha),
                      _Ratio(*self.alpha_min), _Ratio(*self.alpha_max), int(self.n_layers),
                      int(self.coprime_c), int(self.base_max))


_lib = None


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded C library (built in-tree; raises if it cannot be loaded or built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            from ._build import build
            build()
        L = ctypes.CDLL(_LIB_PATH)
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
        sp = ctypes.POINTER(_Sched)
        L.fibattn_offsets.argtypes = [sp, i32, i32, i32, ctypes.POINTER(i32), i32, ctypes.POINTER(i32)]
        L.fibattn_offsets_device.argtypes = [sp, i32, i32, i32, i32, vp, vp, vp]
        L.fibattn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, sp, i32,
                                  i32, vp]
        L.fibattn_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32,
                                      sp, i32, i32, vp]
        u64 = ctypes.c_uint64
        i64 = ctypes.c_int64
        L.fibattn_frac_offsets.argtypes = [f32, i32, i64, i32, i32, ctypes.POINTER(i32),
                                           ctypes.POINTER(f32), i32, ctypes.POINTER(i32)]
        L.fibattn_fwd_frac.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32,
                                       i64, ctypes.POINTER(f32), i32, vp]
        L.fibattn_bwd_frac_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, i64,
                                                      ctypes.POINTER(f32), i32, ctypes.POINTER(u64)]
        L.fibattn_bwd_frac.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, u64, i32, i32,
                                       i32, i32, i32, i32, f32, i32, i64, ctypes.POINTER(f32), i32,
                                       vp]
        L.fibattn_bwd_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, sp, i32, i32,
                                                 ctypes.POINTER(u64)]
        L.fibattn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, u64, i32, i32, i32, i32,
                                  i32, i32, f32, sp, i32, i32, vp]
        L.fibattn_bwd_fused.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, u64, i32, i32, i32,
                                        i32, i32, i32, f32, sp, i32, i32, vp]
        L.fibattn_fwd_bwd_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, sp, i32, i32,
                                                     i32, ctypes.POINTER(u64)]
        L.fibattn_fwd_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, u64, i32, i32, i32,
                                      i32, i32, i32, i32, f32, sp, i32, i32, i32, vp]
        L.fibattn_debug_wait_timeout.argtypes = [i32, vp]
        L.fibattn_debug_wait_timeout.restype = i32
        L.fibattn_rope_table.argtypes = [vp, i32, i32, ctypes.c_double, vp]
        L.fibattn_rope.argtypes = [vp, vp, ctypes.c_int64, i32, i32, i32, vp, i32, i32, vp]
        L.fibattn_fwd_rope.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                       i32, f32, sp, i32, i32, vp, i32, vp]
        L.fibattn_fwd_rope_fused.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                             f32, sp, i32, i32, vp, i32, vp]
        L.fibattn_bwd_rope.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, u64, i32, i32, i32,
                                       i32, i32, i32, i32, f32, sp, i32, i32, vp, i32, vp]
        L.fibattn_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, u64, i32, i32, i32,
                                      i32, i32, i32, i32, f32, sp, i32, i32, vp]
        L.fibattn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                          i32, i32, f32, sp, i32, i32, vp]
        L.fibattn_keyset_debug.argtypes = [sp, i32, i32, i32, vp, vp]
        L.fibattn_poll_device_error.argtypes = [vp]
        L.fibattn_status_string.argtypes = [i32]
        L.fibattn_status_string.restype = ctypes.c_char_p
        L.fibattn_version.restype = i32
        L.fibattn_profile_enable.argtypes = [i32]
        L.fibattn_profile_enable.restype = i32
        L.fibattn_profile_read.argtypes = [ctypes.c_char_p, i32, ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_int64), i32]
        L.fibattn_profile_read.restype = i32
        L.fibattn_last_cuda_error.argtypes = [ctypes.POINTER(ctypes.c_char_p)]
        L.fibattn_last_cuda_error.restype = i32
        L.fibattn_launch_count.argtypes = []
        L.fibattn_launch_count.restype = ctypes.c_int64
        for name in ("fibattn_offsets", "fibattn_offsets_device", "fibattn_fwd", "fibattn_bwd",
                     "fibattn_bwd_workspace_size",
                     "fibattn_bwd_noalloc", "fibattn_keyset_debug", "fibattn_poll_device_error",
                     "fibattn_frac_offsets", "fibattn_fwd_frac", "fibattn_bwd_frac",
                     "fibattn_fwd_gqa", "fibattn_bwd_gqa", "fibattn_rope_table", "fibattn_rope",
                     "fibattn_fwd_rope", "fibattn_bwd_rope", "fibattn_fwd_rope_fused",
                     "fibattn_bwd_frac_workspace_size"):
            getattr(L, name).restype = i32
        _lib = L
    return _lib


def last_cuda_error() -> Tuple[int, str]:
    """(cudaError_t value, failing call) behind the most recent CUDA_ERR status."""
    where = ctypes.c_char_p()
    code = lib().fibattn_last_cuda_error(ctypes.byref(where))
    return int(code), (where.value or b"").decode()


def status_string(status: int) -> str:
    return lib().fibattn_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != OK:
        raise FibAttnError(status, where)


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def offsets(sched: Schedule, layer: int, W: int, T: int) -> list:
    """Host-built offset table of one layer (fibattn_offsets)."""
    cap = MAX_OFFSETS
    buf = (ctypes.c_int32 * cap)()
    n = ctypes.c_int32(0)
    s = sched.to_c()
    _check(lib().fibattn_offsets(ctypes.byref(s), layer, W, T, buf, cap, ctypes.byref(n)),
           "fibattn_offsets")
    return list(buf[: n.value])


def offsets_device(sched: Schedule, layer0: int, n_layers: int, W: int, T: int,
                   device="cuda") -> Tuple[torch.Tensor, torch.Tensor]:
    """Device-built tables [n_layers, MAX_OFFSETS] (-1 padded) and counts [n_layers]."""
    tab = torch.empty((n_layers, MAX_OFFSETS), dtype=torch.int32, device=device)
    cnt = torch.empty((n_layers,), dtype=torch.int32, device=device)
    s = sched.to_c()
    _check(lib().fibattn_offsets_device(ctypes.byref(s), layer0, n_layers, W, T, _ptr(tab),
                                        _ptr(cnt), _stream(tab)), "fibattn_offsets_device")
    return tab, cnt


def _shape(q: torch.Tensor):
    if q.dim() == 5:
        Lc, B, H, T, d = q.shape
    elif q.dim() == 4:
        Lc, (B, H, T, d) = 1, q.shape
    else:
        raise ValueError("q must be [B, H, T, d] or [Lc, B, H, T, d]")
    return Lc, B, H, T, d


def _kv_heads(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor) -> int:
    """H_kv of a grouped-query call: k and v share a shape that differs from q's only in the
    head dim (-3), which divides q's."""
    if k.shape != v.shape or k.dim() != q.dim() or k.dim() < 4:
        raise ValueError("k and v must share a shape with q's rank")
    if k.shape[:-3] != q.shape[:-3] or k.shape[-2:] != q.shape[-2:]:
        raise ValueError("k/v may differ from q only in the head dim")
    H, Hkv = q.shape[-3], k.shape[-3]
    if Hkv < 1 or H % Hkv:
        raise ValueError("q heads must be a multiple of the kv heads")
    return Hkv


def _check_tensors(ref: torch.Tensor, *ts):
    if not ref.is_cuda:
        raise ValueError("tensors must be on a CUDA device (there is no CPU path)")
    if ref.dtype not in _DTYPES:
        raise ValueError("dtype must be float32 or bfloat16")
    if not ref.is_contiguous():
        raise ValueError("tensors must be contiguous")
    for t in ts:
        if t.device != ref.device or t.dtype != ref.dtype or t.shape != ref.shape:
            raise ValueError("q/k/v/o/dO/dq/dk/dv must share device, dtype and shape")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _check_lse(lse: torch.Tensor, q: torch.Tensor):
    # lse is written by the forwards and read by the backwards: one float32 per query row
    if (lse.dtype != torch.float32 or lse.device != q.device
            or tuple(lse.shape) != tuple(q.shape[:-1]) or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 tensor shaped q.shape[:-1] on q's device")


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, W: int, sched: Schedule,
        layer0: int = 0, scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
        lse: Optional[torch.Tensor] = None):
    """Sparse attention forward; returns (o, lse). q/k/v: [Lc,B,H,T,64] or [B,H,T,64]; k and
    v may have fewer heads than q (grouped-query: query head h reads kv head h // (H/H_kv))."""
    Lc, B, H, T, d = _shape(q)
    Hkv = _kv_heads(q, k, v)
    o = torch.empty_like(q) if out is None else out
    _check_tensors(q, o)
    _check_tensors(k, v)
    if k.dtype != q.dtype or k.device != q.device:
        raise ValueError("q/k/v must share device and dtype")
    if lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    s = sched.to_c()
    _check_lse(lse, q)
    st = lib().fibattn_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, T, d,
                               _DTYPES[q.dtype], W, float(scale or 0.0), ctypes.byref(s), layer0,
                               Lc, _stream(q))
    _check(st, "fibattn_fwd_gqa")
    return o, lse


def frac_offsets(alpha: float, W: int, T: int, base: str = "fib", base_max: int = 0):
    """Fractional-offset table of a real alpha (fibattn_frac_offsets): (ceil(d) list, weight
    list) for the distances d = alpha * F kept by the table rule, alpha taken as float32."""
    cap = MAX_OFFSETS
    cbuf = (ctypes.c_int32 * cap)()
    wbuf = (ctypes.c_float * cap)()
    n = ctypes.c_int32(0)
    _check(lib().fibattn_frac_offsets(float(alpha), _BASES[base], int(base_max), W, T, cbuf, wbuf,
                                      cap, ctypes.byref(n)), "fibattn_frac_offsets")
    return list(cbuf[: n.value]), list(wbuf[: n.value])


def fwd_frac(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, W: int, alphas: Sequence[float],
             base: str = "fib", base_max: int = 0, scale: Optional[float] = None,
             out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None):
    """Forward with fractional offsets (learned alphas, one float per call-layer, linear
    interpolation between key/value rows); returns (o, lse)."""
    Lc, B, H, T, d = _shape(q)
    a = _alphas_c(alphas, Lc)
    o = torch.empty_like(q) if out is None else out
    _check_tensors(q, k, v, o)
    if lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    _check_lse(lse, q)
    st = lib().fibattn_fwd_frac(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, T, d,
                                _DTYPES[q.dtype], W, float(scale or 0.0), _BASES[base],
                                int(base_max), a, Lc, _stream(q))
    _check(st, "fibattn_fwd_frac")
    return o, lse


def _alphas_c(alphas, Lc):
    if len(alphas) != Lc:
        raise ValueError("need one alpha per layer of the call")
    return (ctypes.c_float * Lc)(*[float(x) for x in alphas])


def bwd_frac_workspace_size(q: torch.Tensor, W: int, alphas: Sequence[float], base: str = "fib",
                            base_max: int = 0) -> int:
    """Bytes of device workspace bwd_frac() needs for q's shape and dtype."""
    Lc, B, H, T, d = _shape(q)
    if q.dtype not in _DTYPES:
        raise ValueError("dtype must be float32 or bfloat16")
    n = ctypes.c_uint64(0)
    _check(lib().fibattn_bwd_frac_workspace_size(B, H, T, d, _DTYPES[q.dtype], W, _BASES[base],
                                                 int(base_max), _alphas_c(alphas, Lc), Lc,
                                                 ctypes.byref(n)),
           "fibattn_bwd_frac_workspace_size")
    return int(n.value)


def bwd_frac(q, k, v, o, lse, dO, W: int, alphas: Sequence[float], base: str = "fib",
             base_max: int = 0, scale: Optional[float] = None, dq=None, dk=None, dv=None,
             dalpha=None, workspace=None):
    """Backward of fwd_frac; returns (dq, dk, dv, dalpha) with dalpha a float32 [Lc] tensor
    on q's device (the gradient of each layer's alpha)."""
    Lc, B, H, T, d = _shape(q)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    _check_tensors(q, k, v, o, dO, dq, dk, dv)
    if dalpha is None:
        dalpha = torch.empty(Lc, dtype=torch.float32, device=q.device)
    if (dalpha.device != q.device or dalpha.dtype != torch.float32 or dalpha.numel() != Lc
            or not dalpha.is_contiguous()):
        raise ValueError("dalpha must be a contiguous float32 [Lc] tensor on q's device")
    need = bwd_frac_workspace_size(q, W, alphas, base, base_max)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if workspace.device != q.device or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on q's device")
    _check_lse(lse, q)
    st = lib().fibattn_bwd_frac(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                                _ptr(dk), _ptr(dv), _ptr(dalpha), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), B, H, T, d,
                                _DTYPES[q.dtype], W, float(scale or 0.0), _BASES[base],
                                int(base_max), _alphas_c(alphas, Lc), Lc, _stream(q))
    _check(st, "fibattn_bwd_frac")
    return dq, dk, dv, dalpha


def bwd_workspace_size(q: torch.Tensor, W: int, sched: Schedule, layer0: int = 0) -> int:
    """Bytes of device workspace fibattn_bwd needs for tensors shaped like q."""
    Lc, B, H, T, d = _shape(q)
    if q.dtype not in _DTYPES:
        raise ValueError("dtype must be float32 or bfloat16")
    n = ctypes.c_uint64(0)
    s = sched.to_c()
    _check(lib().fibattn_bwd_workspace_size(B, H, T, d, _DTYPES[q.dtype], W, ctypes.byref(s),
                                            layer0, Lc, ctypes.byref(n)),
           "fibattn_bwd_workspace_size")
    return int(n.value)


def bwd(q, k, v, o, lse, dO, W: int, sched: Schedule, layer0: int = 0,
        scale: Optional[float] = None, dq=None, dk=None, dv=None, workspace=None):
    """Sparse attention backward from the saved forward; returns (dq, dk, dv) (dk, dv shaped
    like k, v: grouped-query calls sum each kv row over the heads that read it).
    workspace: optional uint8 device tensor of at least bwd_workspace_size() bytes."""
    Lc, B, H, T, d = _shape(q)
    Hkv = _kv_heads(q, k, v)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(k) if dv is None else dv
    _check_tensors(q, o, dO, dq)
    _check_tensors(k, v, dk, dv)
    if k.dtype != q.dtype or k.device != q.device:
        raise ValueError("q/k/v must share device and dtype")
    need = bwd_workspace_size(q, W, sched, layer0)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if workspace.device != q.device or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on q's device")
    s = sched.to_c()
    _check_lse(lse, q)
    st = lib().fibattn_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                               _ptr(dk), _ptr(dv), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), B, H, Hkv, T, d,
                               _DTYPES[q.dtype], W, float(scale or 0.0), ctypes.byref(s), layer0,
                               Lc, _stream(q))
    _check(st, "fibattn_bwd_gqa")
    return dq, dk, dv


def bwd_fused_workspace_size(q: torch.Tensor) -> int:
    """Bytes of device workspace fibattn_bwd_fused needs for tensors shaped like q: D and
    lse * log2(e), each [Lc][B][H][T_pad] float32 (T_pad = T rounded up to 4), 256-aligned."""
    Lc, B, H, T, d = _shape(q)
    rows = Lc * B * H * ((T + 3) // 4 * 4)
    return 2 * ((rows * 4 + 255) // 256 * 256)


def bwd_fused(q, k, v, o, lse, dO, W: int, sched: Schedule, layer0: int = 0,
              scale: Optional[float] = None, dq=None, dk=None, dv=None, workspace=None):
    """The one-pass backward (fibattn_bwd_fused): one thread block per 128-row tile writes
    dq of its queries and dk, dv of its keys. bf16, head size 64, one kv head per query head.
    Returns (dq, dk, dv), equal to bwd()'s bit for bit. workspace: optional uint8 device
    tensor of at least bwd_fused_workspace_size() bytes."""
    Lc, B, H, T, d = _shape(q)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_tensors(q, k, v, o, dO, dq, dk, dv)
    if workspace is None:
        workspace = torch.empty(bwd_fused_workspace_size(q), dtype=torch.uint8, device=q.device)
    if workspace.device != q.device or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on q's device")
    s = sched.to_c()
    _check_lse(lse, q)
    st = lib().fibattn_bwd_fused(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO),
                                 _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), B, H, T, d,
                                 _DTYPES[q.dtype], W, float(scale or 0.0), ctypes.byref(s),
                                 layer0, Lc, _stream(q))
    _check(st, "fibattn_bwd_fused")
    return dq, dk, dv


def fwd_bwd_workspace_size(q: torch.Tensor, W: int, sched: Schedule, layer0: int = 0,
                           n_streams: int = 2) -> int:
    """Bytes of device workspace fibattn_fwd_bwd needs for tensors shaped like q."""
    Lc, B, H, T, d = _shape(q)
    if q.dtype not in _DTYPES:
        raise ValueError("dtype must be float32 or bfloat16")
    n = ctypes.c_uint64(0)
    s = sched.to_c()
    _check(lib().fibattn_fwd_bwd_workspace_size(B, H, T, d, _DTYPES[q.dtype], W, ctypes.byref(s),
                                                layer0, Lc, int(n_streams), ctypes.byref(n)),
           "fibattn_fwd_bwd_workspace_size")
    return int(n.value)


def fwd_bwd(q, k, v, dO, W: int, sched: Schedule, layer0: int = 0, n_streams: int = 2,
            scale: Optional[float] = None, out=None, lse=None, dq=None, dk=None, dv=None,
            workspace=None):
    """Forward and backward of the layer stack in one call (fibattn_fwd_bwd): the layers are
    split into n_streams groups that run on concurrent streams of the library, forked from and
    joined back into the current stream. Returns (o, lse, dq, dk, dv), equal bit for bit to
    fwd() followed by bwd(). The first call with n_streams > 1 on a device creates the
    library's streams there: make it before any CUDA-graph capture."""
    Lc, B, H, T, d = _shape(q)
    Hkv = _kv_heads(q, k, v)
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device) if lse is None else lse
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_tensors(q, o, dO, dq)
    _check_tensors(k, v, dk, dv)
    if k.dtype != q.dtype or k.device != q.device:
        raise ValueError("q/k/v must share device and dtype")
    need = fwd_bwd_workspace_size(q, W, sched, layer0, n_streams)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if workspace.device != q.device or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on q's device")
    s = sched.to_c()
    _check_lse(lse, q)
    st = lib().fibattn_fwd_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(o), _ptr(lse), _ptr(dq),
                               _ptr(dk), _ptr(dv), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), B, H, Hkv, T, d,
                               _DTYPES[q.dtype], W, float(scale or 0.0), ctypes.byref(s), layer0,
                               Lc, int(n_streams), _stream(q))
    _check(st, "fibattn_fwd_bwd")
    return o, lse, dq, dk, dv


def bwd_noalloc(q, k, v, o, lse, dO, W: int, sched: Schedule, layer0: int = 0,
                scale: Optional[float] = None, dq=None, dk=None, dv=None):
    """Backward for callers that cannot allocate device memory: like bwd(), but the
    workspace is the library's fixed per-device array (fibattn_bwd_noalloc), so none is
    passed. Rejects calls whose workspace exceeds NOALLOC_SCRATCH_BYTES (FibAttnError
    SCRATCH_LIMIT).
    The first call on a device should come before any stream capture; calls whose
    kernels overlap on the GPU share the one scratch array and race."""
    Lc, B, H, T, d = _shape(q)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    _check_tensors(q, k, v, o, dO, dq, dk, dv)
    s = sched.to_c()
    _check_lse(lse, q)
    st = lib().fibattn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO),
                                   _ptr(dq), _ptr(dk), _ptr(dv), B, H, T, d, _DTYPES[q.dtype], W,
                                   float(scale or 0.0), ctypes.byref(s), layer0, Lc, _stream(q))
    _check(st, "fibattn_bwd_noalloc")
    return dq, dk, dv


def keyset_debug(sched: Schedule, layer: int, W: int, T: int, device="cuda") -> torch.Tensor:
    """Device-materialised key sets of one layer as a bool [T, T] tensor (on `device`)."""
    words = (T + 31) // 32
    m = torch.zeros((T, words), dtype=torch.int32, device=device)
    s = sched.to_c()
    _check(lib().fibattn_keyset_debug(ctypes.byref(s), layer, W, T, _ptr(m), _stream(m)),
           "fibattn_keyset_debug")
    bits = (m.unsqueeze(-1) >> torch.arange(32, device=device, dtype=torch.int32)) & 1
    return bits.reshape(T, words * 32)[:, :T].bool()


def poll_device_error(device="cuda"):
    """Synchronise the current stream and raise if a kernel latched an error."""
    st = lib().fibattn_poll_device_error(
        ctypes.c_void_p(torch.cuda.current_stream(torch.device(device)).cuda_stream))
    _check(st, "fibattn_poll_device_error")


class FibSparseAttention(torch.autograd.Function):
    """autograd wrapper: forward and backward both run the library's kernels."""

    @staticmethod
    def forward(ctx, q, k, v, W: int, sched: Schedule, layer0: int = 0, scale=None):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        o, lse = fwd(q, k, v, W, sched, layer0, scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.cfg = (W, sched, layer0, scale)
        return o

    @staticmethod
    def backward(ctx, dO):
        q, k, v, o, lse = ctx.saved_tensors
        W, sched, layer0, scale = ctx.cfg
        dq, dk, dv = bwd(q, k, v, o, lse, dO.contiguous(), W, sched, layer0, scale)
        return dq, dk, dv, None, None, None, None


class FibFracAttention(torch.autograd.Function):
    """autograd wrapper of the fractional-offset (learned-alpha) attention: alpha is a
    float32 tensor [Lc] (on any device; read on the host at every call) and receives its
    gradient from the library's backward."""

    @staticmethod
    def forward(ctx, q, k, v, alpha, W: int, base: str = "fib", base_max: int = 0, scale=None):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        alphas = [float(x) for x in alpha.detach().to("cpu", torch.float32).reshape(-1)]
        o, lse = fwd_frac(q, k, v, W, alphas, base, base_max, scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.cfg = (W, alphas, base, base_max, scale, alpha.shape, alpha.device, alpha.dtype)
        return o

    @staticmethod
    def backward(ctx, dO):
        q, k, v, o, lse = ctx.saved_tensors
        W, alphas, base, base_max, scale, ashape, adev, adtype = ctx.cfg
        dq, dk, dv, da = bwd_frac(q, k, v, o, lse, dO.contiguous(), W, alphas, base, base_max,
                                  scale)
        return dq, dk, dv, da.to(adev, adtype).reshape(ashape), None, None, None, None


def rope_table(T: int, base: float = 10000.0, device="cuda") -> torch.Tensor:
    """cos/sin table of vanilla RoPE for positions 0..T-1 (fibattn_rope_table), a float32
    [T, 32, 2] device tensor; build once per (T, base)."""
    t = torch.empty((T, 32, 2), dtype=torch.float32, device=device)
    _check(lib().fibattn_rope_table(_ptr(t), T, 64, float(base), _stream(t)), "fibattn_rope_table")
    return t


def rope(x: torch.Tensor, table: torch.Tensor, inverse: bool = False,
         out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """x [..., T, 64] with RoPE applied (fibattn_rope); `out` may be x (in place)."""
    if not x.is_cuda or x.dtype not in _DTYPES or not x.is_contiguous() or x.shape[-1] != 64:
        raise ValueError("x must be a contiguous CUDA float32/bfloat16 tensor [..., T, 64]")
    T = x.shape[-2]
    if table.dtype != torch.float32 or table.device != x.device or table.shape[0] < T or \
            not table.is_contiguous():
        raise ValueError("table must be a contiguous float32 rope_table of >= T rows on x's device")
    y = torch.empty_like(x) if out is None else out
    if y.shape != x.shape or y.dtype != x.dtype or y.device != x.device or not y.is_contiguous():
        raise ValueError("out must match x")
    slices = x.numel() // (T * 64)
    _check(lib().fibattn_rope(_ptr(x), _ptr(y), slices, T, 64, _DTYPES[x.dtype], _ptr(table),
                              table.shape[0], int(bool(inverse)), _stream(x)), "fibattn_rope")
    return y


def _check_table(table: torch.Tensor, T: int, ref: torch.Tensor):
    if table.dtype != torch.float32 or table.device != ref.device or table.shape[0] < T or \
            not table.is_contiguous():
        raise ValueError("table must be a contiguous float32 rope_table of >= T rows on q's device")


def fwd_rope(q, k, v, W: int, sched: Schedule, table: torch.Tensor, layer0: int = 0,
             scale: Optional[float] = None, out=None, lse=None, rotated=None):
    """Forward with RoPE on q and k before the gather (fibattn_fwd_rope: q and k rotated, then
    the attention). Returns (o, lse, (q_rot, k_rot)); keep q_rot and k_rot for bwd_rope.
    `rotated` may pass preallocated (q_rot, k_rot) buffers."""
    Lc, B, H, T, d = _shape(q)
    Hkv = _kv_heads(q, k, v)
    qr, kr = rotated if rotated is not None else (torch.empty_like(q), torch.empty_like(k))
    o = torch.empty_like(q) if out is None else out
    _check_tensors(q, o, qr)
    _check_tensors(k, v, kr)
    _check_table(table, T, q)
    if k.dtype != q.dtype or k.device != q.device:
        raise ValueError("q/k/v must share device and dtype")
    if lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    s = sched.to_c()
    _check_lse(lse, q)
    st = lib().fibattn_fwd_rope(_ptr(q), _ptr(k), _ptr(v), _ptr(qr), _ptr(kr), _ptr(o), _ptr(lse),
                                B, H, Hkv, T, d, _DTYPES[q.dtype], W, float(scale or 0.0),
                                ctypes.byref(s), layer0, Lc, _ptr(table), table.shape[0],
                                _stream(q))
    _check(st, "fibattn_fwd_rope")
    return o, lse, (qr, kr)


def fwd_rope_fused(q, k, v, W: int, sched: Schedule, table: torch.Tensor, layer0: int = 0,
                   scale: Optional[float] = None, out=None, lse=None):
    """Forward with RoPE applied inside the attention kernel (fibattn_fwd_rope_fused): q and k
    are read unrotated and no rotated copy is written, for forward-only callers (bf16, d = 64).
    Returns (o, lse); agrees with fwd_rope to rounding."""
    Lc, B, H, T, d = _shape(q)
    Hkv = _kv_heads(q, k, v)
    o = torch.empty_like(q) if out is None else out
    _check_tensors(q, o)
    _check_tensors(k, v)
    _check_table(table, T, q)
    if k.dtype != q.dtype or k.device != q.device:
        raise ValueError("q/k/v must share device and dtype")
    if lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    s = sched.to_c()
    _check_lse(lse, q)
    st = lib().fibattn_fwd_rope_fused(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, T,
                                      d, _DTYPES[q.dtype], W, float(scale or 0.0), ctypes.byref(s),
                                      layer0, Lc, _ptr(table), table.shape[0], _stream(q))
    _check(st, "fibattn_fwd_rope_fused")
    return o, lse


def bwd_rope(q_rot, k_rot, v, o, lse, dO, W: int, sched: Schedule, table: torch.Tensor,
             layer0: int = 0, scale: Optional[float] = None, dq=None, dk=None, dv=None,
             workspace=None):
    """Backward through RoPE from fwd_rope's rotated q and k (fibattn_bwd_rope: dq and dk come
    out rotated back, as the gradients of the unrotated q and k). Returns (dq, dk, dv)."""
    Lc, B, H, T, d = _shape(q_rot)
    Hkv = _kv_heads(q_rot, k_rot, v)
    dq = torch.empty_like(q_rot) if dq is None else dq
    dk = torch.empty_like(k_rot) if dk is None else dk
    dv = torch.empty_like(k_rot) if dv is None else dv
    _check_tensors(q_rot, o, dO, dq)
    _check_tensors(k_rot, v, dk, dv)
    _check_table(table, T, q_rot)
    need = bwd_workspace_size(q_rot, W, sched, layer0)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q_rot.device)
    if workspace.device != q_rot.device or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on q's device")
    s = sched.to_c()
    _check_lse(lse, q_rot)
    st = lib().fibattn_bwd_rope(_ptr(q_rot), _ptr(k_rot), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO),
                                _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), B, H, Hkv, T, d,
                                _DTYPES[q_rot.dtype], W, float(scale or 0.0), ctypes.byref(s),
                                layer0, Lc, _ptr(table), table.shape[0], _stream(q_rot))
    _check(st, "fibattn_bwd_rope")
    return dq, dk, dv


def debug_wait_timeout(limit_ms: int = 50, device="cuda"):
    """Launch the failure-path check (fibattn_debug_wait_timeout): a bounded wait that runs
    out; poll_device_error() afterwards raises FibAttnError with status TIMEOUT."""
    st = lib().fibattn_debug_wait_timeout(
        int(limit_ms), ctypes.c_void_p(torch.cuda.current_stream(torch.device(device)).cuda_stream))
    _check(st, "fibattn_debug_wait_timeout")
