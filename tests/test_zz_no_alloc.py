"""The allocation-free RMSNorm backward, fq_rmsnorm_bwd_noalloc.

It serves callers that cannot allocate device memory or pass a workspace (a plugin whose host
framework owns every device buffer and hands over only tensors; a latency-critical loop that must
never call cudaMalloc). It keeps its dw partial sums in the library's own fixed-size device array
instead. These tests call it through the C ABI and compare it with fq_rmsnorm_bwd (the workspace
entry point) and with the oracle under the parity tolerances, on two calls in a row with different
shapes, so a call that read the previous call's leftovers would show up. This file is named to be
collected last.
"""
import ctypes

import pytest
import torch

from fp8_quant_memory_gb300 import _capi
from fp8_quant_memory_gb300 import workloads as wl
from parity import assert_dw_close, assert_storage_close, assert_within_one_ulp


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, x, w, g, eps=1e-6):
    M, N = x.shape
    dx = torch.empty_like(x)
    dw = torch.empty_like(w)
    dw32 = torch.empty((N,), dtype=torch.float32, device=x.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.fq_rmsnorm_bwd_noalloc(_p(x), _p(w), _p(g), _p(dx), _p(dw), _p(dw32), M, N, _capi.FQ_BF16, eps, stream)
    assert rc == 0, lib.fq_last_error().decode()
    return dx, dw, dw32


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice(orc, cuda_ok):
    import fp8_quant_memory_gb300 as fq

    lib = _capi.load()
    # 8192 x 4096 fills the built-in scratch exactly (256 chunks x 4096 columns x 4 bytes); the
    # second, smaller call reuses the array that the first left behind.
    for M, N, seed in ((8192, 4096, 11), (333, 1024, 12)):
        h = wl.rmsnorm_inputs(M, N, "bf16", seed=seed)
        d = {k: v.cuda() for k, v in h.items()}
        dx, dw, dw32 = _noalloc(lib, d["x"], d["w"], d["g"])
        dx_ref, dw_ref, dw32_ref = fq.rmsnorm_bwd(d["x"], d["w"], d["g"])
        torch.cuda.synchronize()
        assert_storage_close(dx, dx_ref.cpu(), "dx")
        assert_dw_close(dw32, dw32_ref.cpu())
        assert_within_one_ulp(dw, dw_ref.cpu())
        # and against the oracle (the Ch.17 page's RMSNormTileLang.backward)
        dx_o, dw_o, dw32_o = orc.rmsnorm_bwd(h["x"], h["w"], h["g"])
        assert_storage_close(dx, dx_o, "dx (oracle)")
        assert_dw_close(dw32, dw32_o)
        assert_within_one_ulp(dw, dw_o)


def test_noalloc_rejects_problems_beyond_the_scratch():
    """Needs no GPU: the size check runs on the host before anything touches the device."""
    from fp8_quant_memory_gb300 import build

    try:
        build.build()
    except RuntimeError as e:
        pytest.skip(str(e))
    lib = _capi.load()
    p = ctypes.c_void_p(256)
    rc = lib.fq_rmsnorm_bwd_noalloc(p, p, p, p, p, None, 8192, 8192, _capi.FQ_BF16, 1e-6, None)
    assert rc == _capi.FQ_ERR_INVALID_ARG
    assert "scratch" in lib.fq_last_error().decode()
