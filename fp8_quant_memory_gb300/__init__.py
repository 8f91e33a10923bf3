"""fp8_quant_memory_gb300 -- fused RMSNorm -> NeoX partial RoPE -> per-row FP8 (e4m3fn) on GB300.

Thin PyTorch binding over the C ABI in include/fq.h (libfq.so, sm_103a kernels). Each function here
checks tensor devices/dtypes/shapes, allocates outputs with torch when the caller passes none, and
calls the entry point of the same name on the current CUDA stream. Every step of the computation
runs in libfq's kernels; nothing here computes.

Functions (see include/fq.h for the exact definitions and the pages each one follows):
    rmsnorm_fwd(x, w, eps)                                    -> y
    rmsnorm_rope(x, w, cos, sin, eps)                         -> y
    rmsnorm_rope_quant(x, w, cos, sin, eps, fp8_max, want_y)  -> (y | None, q, scale)
    qk_norm_rope_quant(qk, wq, wk, cos, sin, Hq, Hk, ...)     -> (q, scale)
    rmsnorm_bwd(x, w, grad_y, eps)                            -> (dx, dw, dw_f32)
    RMSNormFunction / rmsnorm: autograd wrapper (forward and backward both in libfq)
fp8 outputs are torch.uint8 tensors of e4m3fn codes (``.view(torch.float8_e4m3fn)`` reinterprets).
"""
from __future__ import annotations

import ctypes

import torch

from . import _capi

__all__ = ["layernorm_fwd", "rmsnorm_fwd", "rmsnorm_fwd_rstd", "rmsnorm_bwd_rstd", "rmsnorm_rope", "rmsnorm_rope_quant", "rmsnorm_rope_quant_groups", "qk_norm_rope_quant", "qk_norm_rope_quant_blocks",
           "rmsnorm_bwd",
           "rmsnorm_bwd_workspace_bytes", "rmsnorm", "RMSNormFunction", "device_status", "check_bounded_wait",
           "set_strict",
           "stream_floor", "FqError"]

FqError = _capi.FqError

_DT = {torch.bfloat16: _capi.FQ_BF16, torch.float16: _capi.FQ_FP16, torch.float32: _capi.FQ_FP32}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need_cuda(name: str, *ts):
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name}: every tensor must be on a CUDA device")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name}: tensors are on different devices")
    return dev


def _contig(name: str, **ts):
    for k, t in ts.items():
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name}: {k} must be contiguous")


def _dtype(name: str, t: torch.Tensor) -> int:
    if t.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError(f"{name}: storage dtype must be bfloat16 or float16, got {t.dtype}")
    return _DT[t.dtype]


def _table_dtype(name: str, cos, sin) -> int:
    if cos is None:
        return _capi.FQ_FP32
    if cos.dtype != sin.dtype or cos.dtype not in _DT:
        raise ValueError(f"{name}: cos and sin must share one of bfloat16/float16/float32")
    return _DT[cos.dtype]


def rmsnorm_fwd(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6, out: torch.Tensor | None = None):
    """y = dtype(x * rsqrt(mean(x^2) + eps) * w) over the last dim of a 2-D x."""
    name = "rmsnorm_fwd"
    dev = _need_cuda(name, x, w, out)
    _contig(name, x=x, w=w, out=out)
    M, N = x.shape
    y = torch.empty_like(x) if out is None else out
    _capi.call("fq_rmsnorm_fwd", _ptr(x), _ptr(w), _ptr(y), M, N, _dtype(name, x), eps, _stream(dev))
    return y


def rmsnorm_fwd_rstd(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6, out: torch.Tensor | None = None,
                     rstd: torch.Tensor | None = None):
    """rmsnorm_fwd that also returns each row's fp32 rstd (for rmsnorm_bwd_rstd): (y, rstd [M])."""
    name = "rmsnorm_fwd_rstd"
    dev = _need_cuda(name, x, w, out, rstd)
    _contig(name, x=x, w=w, out=out, rstd=rstd)
    M, N = x.shape
    y = torch.empty_like(x) if out is None else out
    rstd = torch.empty((M,), dtype=torch.float32, device=dev) if rstd is None else rstd
    _capi.call("fq_rmsnorm_fwd_rstd", _ptr(x), _ptr(w), _ptr(y), _ptr(rstd), M, N, _dtype(name, x), eps, _stream(dev))
    return y, rstd


def layernorm_fwd(x: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor | None = None, eps: float = 1e-5,
                  out: torch.Tensor | None = None):
    """y = dtype(((x - mean) * rsqrt(var + eps)) * gamma + beta) over the last dim of a 2-D x."""
    name = "layernorm_fwd"
    dev = _need_cuda(name, x, gamma, beta, out)
    _contig(name, x=x, gamma=gamma, beta=beta, out=out)
    M, N = x.shape
    y = torch.empty_like(x) if out is None else out
    _capi.call("fq_layernorm_fwd", _ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), M, N, _dtype(name, x), eps,
               _stream(dev))
    return y


def rmsnorm_rope(x, w, cos, sin, eps: float = 1e-6, out: torch.Tensor | None = None):
    """RMSNorm then NeoX rotation of the last 2*cos.shape[-1] columns (tables [M, rope_dim/2])."""
    name = "rmsnorm_rope"
    dev = _need_cuda(name, x, w, cos, sin, out)
    _contig(name, x=x, w=w, cos=cos, sin=sin, out=out)
    M, N = x.shape
    R = 2 * cos.shape[-1]
    y = torch.empty_like(x) if out is None else out
    _capi.call("fq_rmsnorm_rope", _ptr(x), _ptr(w), _ptr(cos), _ptr(sin), _ptr(y), M, N, R, _dtype(name, x),
               _table_dtype(name, cos, sin), eps, _stream(dev))
    return y


def rmsnorm_rope_quant(x, w, cos, sin, eps: float = 1e-6, fp8_max: float = 448.0, want_y: bool = True,
                       y: torch.Tensor | None = None, q: torch.Tensor | None = None,
                       scale: torch.Tensor | None = None):
    """RMSNorm + NeoX partial RoPE + per-row FP8. Returns (y or None, q uint8 [M,N], scale fp32 [M])."""
    name = "rmsnorm_rope_quant"
    dev = _need_cuda(name, x, w, cos, sin, y, q, scale)
    _contig(name, x=x, w=w, cos=cos, sin=sin, y=y, q=q, scale=scale)
    M, N = x.shape
    R = 2 * cos.shape[-1]
    if y is None and want_y:
        y = torch.empty_like(x)
    q = torch.empty((M, N), dtype=torch.uint8, device=dev) if q is None else q
    scale = torch.empty((M,), dtype=torch.float32, device=dev) if scale is None else scale
    _capi.call("fq_rmsnorm_rope_quant", _ptr(x), _ptr(w), _ptr(cos), _ptr(sin), _ptr(y), _ptr(q), _ptr(scale),
               M, N, R, _dtype(name, x), _table_dtype(name, cos, sin), eps, fp8_max, _stream(dev))
    return y, q, scale


def rmsnorm_rope_quant_groups(x, w, cos, sin, group_size: int, eps: float = 1e-6, fp8_max: float = 448.0,
                              want_y: bool = True, y: torch.Tensor | None = None, q: torch.Tensor | None = None,
                              scale: torch.Tensor | None = None):
    """RMSNorm + NeoX partial RoPE + FP8 with one scale per group_size columns.
    Returns (y or None, q uint8 [M,N], scale fp32 [M, N // group_size])."""
    name = "rmsnorm_rope_quant_groups"
    dev = _need_cuda(name, x, w, cos, sin, y, q, scale)
    _contig(name, x=x, w=w, cos=cos, sin=sin, y=y, q=q, scale=scale)
    M, N = x.shape
    R = 2 * cos.shape[-1]
    if group_size < 1 or N % group_size != 0:
        raise ValueError(f"{name}: group_size must divide N (N={N}, group_size={group_size})")
    if y is None and want_y:
        y = torch.empty_like(x)
    q = torch.empty((M, N), dtype=torch.uint8, device=dev) if q is None else q
    scale = torch.empty((M, N // group_size), dtype=torch.float32, device=dev) if scale is None else scale
    _capi.call("fq_rmsnorm_rope_quant_groups", _ptr(x), _ptr(w), _ptr(cos), _ptr(sin), _ptr(y), _ptr(q),
               _ptr(scale), M, N, R, group_size, _dtype(name, x), _table_dtype(name, cos, sin), eps, fp8_max,
               _stream(dev))
    return y, q, scale


def qk_norm_rope_quant(qk, wq, wk, cos, sin, Hq: int, Hk: int, eps: float = 1e-6, fp8_max: float = 448.0,
                       rope_dim: int | None = None, q_out: torch.Tensor | None = None,
                       scale: torch.Tensor | None = None):
    """QK-Norm + RoPE + FP8 prologue.

    qk: [T, Hq+Hk, D] or [T, S] (S >= (Hq+Hk)*D, heads packed first; a row stride also works:
    any 2-D/3-D tensor whose last dims are contiguous). Returns (q uint8 [T, H, D], scale fp32 [T, H]).
    """
    name = "qk_norm_rope_quant"
    dev = _need_cuda(name, qk, wq, wk, cos, sin, q_out, scale)
    _contig(name, wq=wq, wk=wk, cos=cos, sin=sin, q_out=q_out, scale=scale)
    H = Hq + Hk
    D = wq.shape[0]
    T = qk.shape[0]
    if qk.dim() == 3:
        if tuple(qk.shape[1:]) != (H, D) or qk.stride(2) != 1 or qk.stride(1) != D:
            raise ValueError(f"{name}: qk must be [T, Hq+Hk, D] with contiguous heads")
    elif qk.dim() == 2:
        if qk.shape[1] < H * D or qk.stride(1) != 1:
            raise ValueError(f"{name}: qk rows must hold (Hq+Hk)*D contiguous elements")
    else:
        raise ValueError(f"{name}: qk must be 2-D or 3-D")
    token_stride = qk.stride(0)
    R = D if rope_dim is None else rope_dim
    q_out = torch.empty((T, H, D), dtype=torch.uint8, device=dev) if q_out is None else q_out
    scale = torch.empty((T, H), dtype=torch.float32, device=dev) if scale is None else scale
    _capi.call("fq_qk_norm_rope_quant", _ptr(qk), token_stride, _ptr(wq), _ptr(wk), _ptr(cos), _ptr(sin),
               _ptr(q_out), _ptr(scale), T, Hq, Hk, D, R, _dtype(name, qk), _table_dtype(name, cos, sin), eps,
               fp8_max, _stream(dev))
    return q_out, scale


def qk_norm_rope_quant_blocks(qk, wq, wk, cos, sin, Hq: int, Hk: int, rows_per_block: int, eps: float = 1e-6,
                              fp8_max: float = 448.0, q_out: torch.Tensor | None = None,
                              scale: torch.Tensor | None = None):
    """The prologue as the Ch.28 page's designs A / B / C: one CTA per block of rows_per_block rows
    (1, 8, Hq + Hk). qk: [T, Hq+Hk, D] packed. Returns (q uint8 [T, H, D], scale fp32 [T, H])."""
    name = "qk_norm_rope_quant_blocks"
    dev = _need_cuda(name, qk, wq, wk, cos, sin, q_out, scale)
    _contig(name, qk=qk, wq=wq, wk=wk, cos=cos, sin=sin, q_out=q_out, scale=scale)
    H = Hq + Hk
    D = wq.shape[0]
    T = qk.shape[0]
    q_out = torch.empty((T, H, D), dtype=torch.uint8, device=dev) if q_out is None else q_out
    scale = torch.empty((T, H), dtype=torch.float32, device=dev) if scale is None else scale
    _capi.call("fq_qk_norm_rope_quant_blocks", _ptr(qk), H * D, _ptr(wq), _ptr(wk), _ptr(cos), _ptr(sin),
               _ptr(q_out), _ptr(scale), T, Hq, Hk, D, D, rows_per_block, _dtype(name, qk),
               _table_dtype(name, cos, sin), eps, fp8_max, _stream(dev))
    return q_out, scale


def rmsnorm_bwd_workspace_bytes(M: int, N: int) -> int:
    return int(_capi.load().fq_rmsnorm_bwd_workspace_bytes(M, N))


def rmsnorm_bwd(x, w, grad_y, eps: float = 1e-6, workspace: torch.Tensor | None = None,
                want_dw_f32: bool = True):
    """RMSNorm backward (rstd recomputed). Returns (dx, dw, dw_f32 or None)."""
    name = "rmsnorm_bwd"
    dev = _need_cuda(name, x, w, grad_y, workspace)
    _contig(name, x=x, w=w, grad_y=grad_y, workspace=workspace)
    M, N = x.shape
    dx = torch.empty_like(x)
    dw = torch.empty_like(w)
    dw32 = torch.empty((N,), dtype=torch.float32, device=dev) if want_dw_f32 else None
    need = rmsnorm_bwd_workspace_bytes(M, N)
    if workspace is None:
        workspace = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
    _capi.call("fq_rmsnorm_bwd", _ptr(x), _ptr(w), _ptr(grad_y), _ptr(dx), _ptr(dw), _ptr(dw32), _ptr(workspace),
               workspace.numel() * workspace.element_size(), M, N, _dtype(name, x), eps, _stream(dev))
    return dx, dw, dw32


def rmsnorm_bwd_rstd(x, w, grad_y, rstd, workspace: torch.Tensor | None = None, want_dw_f32: bool = True):
    """RMSNorm backward with the forward's saved rstd [M] fp32. Returns (dx, dw, dw_f32 or None)."""
    name = "rmsnorm_bwd_rstd"
    dev = _need_cuda(name, x, w, grad_y, rstd, workspace)
    _contig(name, x=x, w=w, grad_y=grad_y, rstd=rstd, workspace=workspace)
    M, N = x.shape
    dx = torch.empty_like(x)
    dw = torch.empty_like(w)
    dw32 = torch.empty((N,), dtype=torch.float32, device=dev) if want_dw_f32 else None
    need = rmsnorm_bwd_workspace_bytes(M, N)
    if workspace is None:
        workspace = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
    _capi.call("fq_rmsnorm_bwd_rstd", _ptr(x), _ptr(w), _ptr(grad_y), _ptr(rstd), _ptr(dx), _ptr(dw), _ptr(dw32),
               _ptr(workspace), workspace.numel() * workspace.element_size(), M, N, _dtype(name, x), _stream(dev))
    return dx, dw, dw32


def device_status(clear: bool = True, device=None) -> int:
    """The device status word (bit 0: a pipelined kernel gave up on a bounded wait)."""
    word = ctypes.c_uint(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _capi.call("fq_device_status", ctypes.byref(word), 1 if clear else 0, _stream(dev))
    return int(word.value)


def set_strict(on: bool) -> bool:
    """Strict mode on or off (returns the previous setting): every call then waits for its stream and
    raises FqError (status FQ_ERR_DEVICE) if a pipelined kernel gave up on a bounded wait."""
    return bool(_capi.load().fq_set_strict(1 if on else 0))


def check_bounded_wait(limit_ms: int = 50, device=None) -> int:
    """Run the bounded-wait diagnostic (a wait that can only give up after limit_ms) and return the
    device status word it leaves (bit 0 set means the wait gave up as designed); clears it."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    device_status(clear=True, device=dev)
    _capi.call("fq_check_bounded_wait", ctypes.c_uint(limit_ms), _stream(dev))
    return device_status(clear=True, device=dev)


def stream_floor(inp: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """The size-matched streaming floor (a measurement aid, not a step of the method): `inp` is a
    contiguous device tensor whose byte size is a multiple of 16; returns (or fills) a uint8 tensor of
    half that size whose 8-byte word i is the XOR of the two 8-byte halves of 16-byte vector i."""
    if not (inp.is_cuda and inp.is_contiguous()):
        raise ValueError("stream_floor: inp must be a contiguous CUDA tensor")
    nbytes = inp.numel() * inp.element_size()
    if nbytes % 16:
        raise ValueError("stream_floor: the input size must be a multiple of 16 bytes")
    n16 = nbytes // 16
    if out is None:
        out = torch.empty(n16 * 8, dtype=torch.uint8, device=inp.device)
    elif not (out.is_cuda and out.is_contiguous() and out.numel() * out.element_size() == n16 * 8):
        raise ValueError("stream_floor: out must be a contiguous CUDA tensor of half the input's bytes")
    _capi.call("fq_stream_floor", _ptr(inp), _ptr(out), n16, _stream(inp.device))
    return out


class RMSNormFunction(torch.autograd.Function):
    """RMSNorm with both directions in libfq ("rmsnorm_tl.py" (Ch.17), RMSNormTileLang): the forward
    saves x and w and the backward recomputes rstd, as the page does; with save_rstd the forward also
    saves its fp32 rstd (4 bytes per row) and the backward reuses it."""

    @staticmethod
    def forward(ctx, x, w, eps, save_rstd=False):
        shape = x.shape
        x2 = x.reshape(-1, shape[-1]).contiguous()
        if save_rstd:
            y, rstd = rmsnorm_fwd_rstd(x2, w.contiguous(), eps)
            ctx.save_for_backward(x2, w, rstd)
        else:
            y = rmsnorm_fwd(x2, w.contiguous(), eps)
            ctx.save_for_backward(x2, w)
        ctx.eps = eps
        ctx.shape = shape
        return y.view(shape)

    @staticmethod
    def backward(ctx, gy):
        saved = ctx.saved_tensors
        x2, w = saved[0], saved[1]
        g2 = gy.reshape(-1, x2.shape[-1]).contiguous()
        if len(saved) == 3:
            dx, dw, _ = rmsnorm_bwd_rstd(x2, w.contiguous(), g2, saved[2], want_dw_f32=False)
        else:
            dx, dw, _ = rmsnorm_bwd(x2, w.contiguous(), g2, ctx.eps, want_dw_f32=False)
        return dx.view(ctx.shape), dw, None, None


def rmsnorm(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6, save_rstd: bool = False) -> torch.Tensor:
    return RMSNormFunction.apply(x, w, eps, save_rstd)
