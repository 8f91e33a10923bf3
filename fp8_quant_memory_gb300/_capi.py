"""ctypes view of libfq (include/fq.h): loads the in-tree library and declares every entry point.

The library must have been built (``python -c "import __graft_entry__ as g; g.build()"`` or
``python fp8_quant_memory_gb300/build.py``); if it is missing, loading raises. There is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

FQ_OK, FQ_ERR_INVALID_ARG, FQ_ERR_UNSUPPORTED, FQ_ERR_MISALIGNED, FQ_ERR_CUDA, FQ_ERR_DEVICE = range(6)
FQ_BF16, FQ_FP16, FQ_FP32 = 0, 1, 2

_vp, _i64, _int, _f32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t

# name -> (restype, argtypes), mirroring include/fq.h
SIGNATURES = {
    "fq_last_error": (ctypes.c_char_p, []),
    "fq_version": (_int, []),
    "fq_device_status": (_int, [ctypes.POINTER(ctypes.c_uint), _int, _vp]),
    "fq_check_bounded_wait": (_int, [ctypes.c_uint, _vp]),
    "fq_set_strict": (_int, [_int]),
    "fq_stream_floor": (_int, [_vp, _vp, _i64, _vp]),
    "fq_rmsnorm_fwd": (_int, [_vp, _vp, _vp, _i64, _i64, _int, _f32, _vp]),
    "fq_rmsnorm_fwd_rstd": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _int, _f32, _vp]),
    "fq_layernorm_fwd": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _int, _f32, _vp]),
    "fq_rmsnorm_rope": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _f32, _vp]),
    "fq_rmsnorm_rope_quant": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _f32,
                                     _f32, _vp]),
    "fq_rmsnorm_rope_quant_groups": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _int,
                                            _int, _f32, _f32, _vp]),
    "fq_qk_norm_rope_quant": (_int, [_vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                     _int, _int, _f32, _f32, _vp]),
    "fq_qk_norm_rope_quant_blocks": (_int, [_vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                            _i64, _int, _int, _f32, _f32, _vp]),
    "fq_rmsnorm_bwd_workspace_bytes": (_sz, [_i64, _i64]),
    "fq_rmsnorm_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64, _int, _f32, _vp]),
    "fq_rmsnorm_bwd_rstd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64, _int, _vp]),
    "fq_rmsnorm_bwd_noalloc": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _f32, _vp]),
}

_lib = None
_lock = threading.Lock()


class FqError(RuntimeError):
    """A libfq entry point returned an error status."""

    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn} failed with status {status}: {message}")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libfq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libfq is not built ({path} missing): run "
                    "`python -c \"import __graft_entry__ as g; g.build()\"` on a machine with nvcc")
            handle = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def call(name: str, *args) -> None:
    """Call an entry point that returns a status; raise FqError on failure."""
    lib = load()
    rc = getattr(lib, name)(*args)
    if rc != FQ_OK:
        msg = lib.fq_last_error()
        raise FqError(name, rc, msg.decode() if msg else "")


def last_error() -> str:
    msg = load().fq_last_error()
    return msg.decode() if msg else ""
