"""Reference oracle for the fused RMSNorm -> NeoX RoPE -> per-row FP8 path (CPU, single thread).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` are the only callers. The product path never imports this package.

This module only marshals torch CPU tensors into the plain C++ loops of ``fq_oracle.cpp`` (which
cites the passages each function restates) and allocates their outputs. It adds no arithmetic.

Storage conventions: bf16 / fp16 tensors are passed as their 16-bit patterns, fp8 results come back
as ``torch.uint8`` e4m3fn codes, scales as ``torch.float32``.
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import build as _build

_FMT = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}
_lib = None
_lock = threading.Lock()

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_f32 = ctypes.c_float
_f64 = ctypes.c_double

_SIGS = {
    "or_encode": [_int, _vp, _vp, _i64],
    "or_decode": [_int, _vp, _vp, _i64],
    "or_rmsnorm_fwd": [_vp, _vp, _vp, _i64, _i64, _int, _f32],
    "or_rmsnorm_rope": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _f32],
    "or_rmsnorm_rope_quant": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _f32, _f32],
    "or_quant_rows": [_vp, _vp, _vp, _i64, _i64, _int, _f32],
    "or_rmsnorm_rope_quant_groups": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _int, _int,
                                     _f32, _f32],
    "or_quant_groups": [_vp, _vp, _vp, _i64, _i64, _i64, _int, _f32],
    "or_qk_norm_rope_quant": [_vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                              _int, _int, _f32, _f32],
    "or_rmsnorm_bwd": [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _f32],
    "or_rmsnorm_bwd_rstd": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int],
    "or_rmsnorm_fwd_rstd": [_vp, _vp, _vp, _vp, _i64, _i64, _int, _f32],
    "or_rmsnorm_f64": [_vp, _vp, _vp, _i64, _i64, _f64],
    "or_layernorm_fwd": [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _f32],
    "or_layernorm_f64": [_vp, _vp, _vp, _vp, _i64, _i64, _f64],
    "or_rope_f64": [_vp, _vp, _vp, _i64, _i64, _i64],
    "or_rmsnorm_bwd_f64": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _f64],
}


def lib() -> ctypes.CDLL:
    """Load (building first if needed) the oracle shared library."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            handle = ctypes.CDLL(path)
            for name, args in _SIGS.items():
                fn = getattr(handle, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            _lib = handle
    return _lib


def _p(t: torch.Tensor | None):
    if t is None:
        return None
    assert t.device.type == "cpu" and t.is_contiguous(), "oracle takes contiguous CPU tensors"
    return ctypes.c_void_p(t.data_ptr())


def _check(rc: int, name: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {name}: invalid arguments (status {rc})")


# ------------------------------------------------------------------ formats
def encode(values: torch.Tensor, dtype) -> torch.Tensor:
    """fp32 values -> bit patterns of ``dtype`` (bf16/fp16 as int16 view, 'e4m3' as uint8)."""
    v = values.to(torch.float32).contiguous()
    if dtype == "e4m3":
        out = torch.empty(v.shape, dtype=torch.uint8)
        fmt = 3
    else:
        out = torch.empty(v.shape, dtype=dtype)
        fmt = _FMT[dtype]
    _check(lib().or_encode(fmt, _p(v), _p(out), v.numel()), "encode")
    return out


def decode(codes: torch.Tensor, dtype=None) -> torch.Tensor:
    """Stored values (bf16/fp16 tensor, or uint8 e4m3fn codes) -> exact fp32 values."""
    c = codes.contiguous()
    fmt = 3 if c.dtype == torch.uint8 else _FMT[c.dtype]
    out = torch.empty(c.shape, dtype=torch.float32)
    _check(lib().or_decode(fmt, _p(c), _p(out), c.numel()), "decode")
    return out


# ------------------------------------------------------------------ forward path
def rmsnorm_fwd(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6) -> torch.Tensor:
    M, N = x.shape
    y = torch.empty_like(x)
    _check(lib().or_rmsnorm_fwd(_p(x), _p(w), _p(y), M, N, _FMT[x.dtype], eps), "rmsnorm_fwd")
    return y


def rmsnorm_fwd_rstd(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6):
    """Forward that also returns each row's fp32 rstd: (y, rstd [M])."""
    M, N = x.shape
    y = torch.empty_like(x)
    rstd = torch.empty((M,), dtype=torch.float32)
    _check(lib().or_rmsnorm_fwd_rstd(_p(x), _p(w), _p(y), _p(rstd), M, N, _FMT[x.dtype], eps), "rmsnorm_fwd_rstd")
    return y, rstd


def rmsnorm_rope(x, w, cos, sin, eps: float = 1e-6) -> torch.Tensor:
    M, N = x.shape
    R = 2 * cos.shape[-1]
    y = torch.empty_like(x)
    _check(lib().or_rmsnorm_rope(_p(x), _p(w), _p(cos), _p(sin), _p(y), M, N, R, _FMT[x.dtype],
                                 _FMT[cos.dtype], eps), "rmsnorm_rope")
    return y


def rmsnorm_rope_quant(x, w, cos, sin, eps: float = 1e-6, fp8_max: float = 448.0, want_y: bool = True):
    """Returns (y or None, q uint8 [M,N], scale fp32 [M])."""
    M, N = x.shape
    R = 2 * cos.shape[-1]
    y = torch.empty_like(x) if want_y else None
    q = torch.empty((M, N), dtype=torch.uint8)
    scale = torch.empty((M,), dtype=torch.float32)
    _check(lib().or_rmsnorm_rope_quant(_p(x), _p(w), _p(cos), _p(sin), _p(y), _p(q), _p(scale), M, N,
                                       R, _FMT[x.dtype], _FMT[cos.dtype], eps, fp8_max),
           "rmsnorm_rope_quant")
    return y, q, scale


def quant_rows(y: torch.Tensor, fp8_max: float = 448.0):
    """Steps a6-a8 alone on rows of a stored y: (q uint8, scale fp32)."""
    M, N = y.shape
    q = torch.empty((M, N), dtype=torch.uint8)
    scale = torch.empty((M,), dtype=torch.float32)
    _check(lib().or_quant_rows(_p(y.contiguous()), _p(q), _p(scale), M, N, _FMT[y.dtype], fp8_max),
           "quant_rows")
    return q, scale


def rmsnorm_rope_quant_groups(x, w, cos, sin, group_size: int, eps: float = 1e-6, fp8_max: float = 448.0,
                              want_y: bool = True):
    """Group-wise scales: returns (y or None, q uint8 [M,N], scale fp32 [M, N/group_size])."""
    M, N = x.shape
    R = 2 * cos.shape[-1]
    y = torch.empty_like(x) if want_y else None
    q = torch.empty((M, N), dtype=torch.uint8)
    scale = torch.empty((M, N // group_size), dtype=torch.float32)
    _check(lib().or_rmsnorm_rope_quant_groups(_p(x), _p(w), _p(cos), _p(sin), _p(y), _p(q), _p(scale), M, N,
                                              R, group_size, _FMT[x.dtype], _FMT[cos.dtype], eps, fp8_max),
           "rmsnorm_rope_quant_groups")
    return y, q, scale


def quant_groups(y: torch.Tensor, group_size: int, fp8_max: float = 448.0):
    """The group-wise quantiser alone on rows of a stored y: (q uint8 [M,N], scale fp32 [M, N/gs])."""
    M, N = y.shape
    q = torch.empty((M, N), dtype=torch.uint8)
    scale = torch.empty((M, N // group_size), dtype=torch.float32)
    _check(lib().or_quant_groups(_p(y.contiguous()), _p(q), _p(scale), M, N, group_size, _FMT[y.dtype],
                                 fp8_max), "quant_groups")
    return q, scale


def qk_norm_rope_quant(qk, wq, wk, cos, sin, hq: int, hk: int, eps: float = 1e-6,
                       fp8_max: float = 448.0, rope_dim: int | None = None):
    """qk: [T, Hq+Hk, D] (or [T, S] with S >= (Hq+Hk)*D, heads packed first). Returns (q, scale)."""
    T = qk.shape[0]
    H = hq + hk
    D = wq.shape[0]
    if not qk.is_contiguous():
        raise ValueError("oracle qk must be contiguous (use a wider 2-D row for a token stride)")
    if qk.dim() == 3:
        if tuple(qk.shape[1:]) != (H, D):
            raise ValueError("qk must be [T, Hq+Hk, D]")
        token_stride = H * D
    elif qk.dim() == 2:
        token_stride = qk.shape[1]
    else:
        raise ValueError("qk must be [T, Hq+Hk, D] or [T, token_stride]")
    R = D if rope_dim is None else rope_dim
    q = torch.empty((T, H, D), dtype=torch.uint8)
    scale = torch.empty((T, H), dtype=torch.float32)
    _check(lib().or_qk_norm_rope_quant(_p(qk), token_stride, _p(wq), _p(wk), _p(cos), _p(sin), _p(q),
                                       _p(scale), T, hq, hk, D, R, _FMT[qk.dtype], _FMT[cos.dtype],
                                       eps, fp8_max), "qk_norm_rope_quant")
    return q, scale


def qk_norm_rope_quant_rounded(qk, wq, wk, cos, sin, hq: int, hk: int, eps: float = 1e-6,
                               fp8_max: float = 448.0):
    """The prologue under the other reading of its cast points: the fusion page's definition
    ("rmsnorm_rope_quant.py", torch_reference_fused) rounds the normalised row and the rotated row to
    the storage dtype, where the prologue statement ("case_norm_rope_quant.py", module docstring)
    names no intermediates and qk_norm_rope_quant keeps fp32 from load to quantiser. Composed from
    rmsnorm_rope_quant: every (token, head) row with its head's weight (wq for the first hq heads,
    wk for the rest) and its token's cos/sin row. qk: contiguous [T, hq+hk, D]. Returns (q, scale)."""
    T, H, D = qk.shape
    if H != hq + hk or not qk.is_contiguous():
        raise ValueError("qk must be a contiguous [T, hq+hk, D]")
    q = torch.empty((T, H, D), dtype=torch.uint8)
    scale = torch.empty((T, H), dtype=torch.float32)
    for h0, h1, w in ((0, hq, wq), (hq, H, wk)):
        nh = h1 - h0
        if nh == 0:
            continue
        x = qk[:, h0:h1].reshape(T * nh, D).contiguous()
        c = cos.repeat_interleave(nh, dim=0).contiguous()  # row t*nh + j: token t's table row
        s = sin.repeat_interleave(nh, dim=0).contiguous()
        _, qq, ss = rmsnorm_rope_quant(x, w, c, s, eps, fp8_max, want_y=False)
        q[:, h0:h1] = qq.view(T, nh, D)
        scale[:, h0:h1] = ss.view(T, nh)
    return q, scale


# ------------------------------------------------------------------ backward
def rmsnorm_bwd(x, w, g, eps: float = 1e-6):
    """Returns (dx, dw, dw_f32)."""
    M, N = x.shape
    dx = torch.empty_like(x)
    dw = torch.empty_like(w)
    dw32 = torch.empty((N,), dtype=torch.float32)
    _check(lib().or_rmsnorm_bwd(_p(x), _p(w), _p(g), _p(dx), _p(dw), _p(dw32), M, N, _FMT[x.dtype], eps),
           "rmsnorm_bwd")
    return dx, dw, dw32


def rmsnorm_bwd_rstd(x, w, g, rstd):
    """Backward with a saved rstd [M] fp32: (dx, dw, dw_f32)."""
    M, N = x.shape
    dx = torch.empty_like(x)
    dw = torch.empty_like(w)
    dw32 = torch.empty((N,), dtype=torch.float32)
    _check(lib().or_rmsnorm_bwd_rstd(_p(x), _p(w), _p(g), _p(rstd.contiguous()), _p(dx), _p(dw), _p(dw32), M, N,
                                     _FMT[x.dtype]), "rmsnorm_bwd_rstd")
    return dx, dw, dw32


def layernorm_fwd(x, g, b=None, eps: float = 1e-5):
    """LayerNorm forward: returns (y, mean fp32 [M], rstd fp32 [M])."""
    M, N = x.shape
    y = torch.empty_like(x)
    mean = torch.empty((M,), dtype=torch.float32)
    rstd = torch.empty((M,), dtype=torch.float32)
    _check(lib().or_layernorm_fwd(_p(x), _p(g), _p(b), _p(y), _p(mean), _p(rstd), M, N, _FMT[x.dtype], eps),
           "layernorm_fwd")
    return y, mean, rstd


# ------------------------------------------------------------------ fp64 twins (pins only)
def layernorm_f64(x, g, b, eps: float):
    x = x.double().contiguous()
    M, N = x.shape
    y = torch.empty_like(x)
    gg = g.double().contiguous()
    bb = None if b is None else b.double().contiguous()
    _check(lib().or_layernorm_f64(_p(x), _p(gg), _p(bb), _p(y), M, N, eps), "layernorm_f64")
    return y


def rmsnorm_f64(x, w, eps: float):
    x = x.to(torch.float64).contiguous()
    w = w.to(torch.float64).contiguous()
    M, N = x.shape
    y = torch.empty_like(x)
    _check(lib().or_rmsnorm_f64(_p(x), _p(w), _p(y), M, N, eps), "rmsnorm_f64")
    return y


def rope_f64(rows, cos, sin):
    rows = rows.to(torch.float64).contiguous().clone()
    cos = cos.to(torch.float64).contiguous()
    sin = sin.to(torch.float64).contiguous()
    M, N = rows.shape
    R = 2 * cos.shape[-1]
    _check(lib().or_rope_f64(_p(rows), _p(cos), _p(sin), M, N, R), "rope_f64")
    return rows


def rmsnorm_bwd_f64(x, w, g, eps: float):
    x = x.to(torch.float64).contiguous()
    w = w.to(torch.float64).contiguous()
    g = g.to(torch.float64).contiguous()
    M, N = x.shape
    dx = torch.empty_like(x)
    dw = torch.empty((N,), dtype=torch.float64)
    _check(lib().or_rmsnorm_bwd_f64(_p(x), _p(w), _p(g), _p(dx), _p(dw), M, N, eps), "rmsnorm_bwd_f64")
    return dx, dw
