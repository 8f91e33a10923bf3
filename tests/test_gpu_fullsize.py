"""GPU parity at the full sizes of the measured workloads, through the same entry points and launch
configuration the benchmark times.

- qk_prologue_4k (4096 tokens x 40 heads x 128), rmsnorm_8k_4k (fwd and bwd) and rope_fp16_64k:
  every output element against the oracle.
- qk_prologue_32k (32768 tokens x 72 heads x 128, 1% outliers x50, positions up to 131072): every
  row against the oracle, plus properties that hold for every row at any size (the amax element of
  each row lands on +-448, scales positive and finite, no NaN codes).
- rope_quant_tiny: y, codes and scales against the oracle (scales within 1e-5 on every row).
"""
import numpy as np
import pytest
import torch

import fp8_quant_memory_gb300 as fq
from fp8_quant_memory_gb300 import workloads as wl
from parity import (assert_own_quantiser, assert_codes_close, assert_dw_close, assert_rope_close, assert_scale_close,
                    assert_storage_close, assert_within_one_ulp, oracle_prologue_parallel,
                    scale_rows_by_own_y)

pytestmark = pytest.mark.gpu


def _cuda(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _row_properties(q: torch.Tensor, scale: torch.Tensor):
    mag = (q & 0x7F)
    assert int((mag == 0x7F).sum()) == 0, "NaN codes"
    assert bool((mag.amax(-1) == 0x7E).all()), "a row whose amax element is not at +-448"
    s = scale
    assert bool(torch.isfinite(s).all()) and bool((s > 0).all())


def test_qk_prologue_4k_full(orc, cuda_ok):
    d = wl.WORKLOADS["qk_prologue_4k"].make()
    q_ref, s_ref = orc.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], 32, 8)
    g = _cuda(d)
    q, s = fq.qk_norm_rope_quant(g["qk"], g["wq"], g["wk"], g["cos"], g["sin"], 32, 8)
    torch.cuda.synchronize()
    assert_scale_close(s, s_ref)
    assert_codes_close(q, q_ref)
    _row_properties(q, s)
    assert fq.device_status(clear=True) == 0


def test_qk_prologue_32k_full(orc, cuda_ok):
    """Every one of the 2,359,296 rows against the oracle (the oracle runs over token slices on a
    thread pool: it is a C library called through ctypes, with no global state)."""
    d = wl.WORKLOADS["qk_prologue_32k"].make()
    g = _cuda(d)
    q, s = fq.qk_norm_rope_quant(g["qk"], g["wq"], g["wk"], g["cos"], g["sin"], 64, 8)
    torch.cuda.synchronize()
    _row_properties(q, s)
    q_ref, s_ref = oracle_prologue_parallel(orc, d, 64, 8)
    assert_scale_close(s, s_ref)
    assert_codes_close(q, q_ref)
    assert fq.device_status(clear=True) == 0


def test_rmsnorm_8k_4k_full(orc, cuda_ok):
    d = wl.WORKLOADS["rmsnorm_8k_4k"].make()
    g = _cuda(d)
    y = fq.rmsnorm_fwd(g["x"], g["w"])
    dx, dw, dw32 = fq.rmsnorm_bwd(g["x"], g["w"], g["g"])
    torch.cuda.synchronize()
    assert_storage_close(y, orc.rmsnorm_fwd(d["x"], d["w"]))
    dx_ref, dw_ref, dw32_ref = orc.rmsnorm_bwd(d["x"], d["w"], d["g"])
    assert_storage_close(dx, dx_ref, "dx")
    assert_dw_close(dw32, dw32_ref)
    assert_within_one_ulp(dw, dw_ref)


def test_rope_fp16_64k_full(orc, cuda_ok):
    d = wl.WORKLOADS["rope_fp16_64k"].make()
    g = _cuda(d)
    y = fq.rmsnorm_rope(g["x"], g["w"], g["cos"], g["sin"])
    torch.cuda.synchronize()
    assert_rope_close(y, orc.rmsnorm_rope(d["x"], d["w"], d["cos"], d["sin"]), orc.rmsnorm_fwd(d["x"], d["w"]),
                      d["cos"], d["sin"])


def test_rope_quant_tiny_full(orc, cuda_ok):
    d = wl.WORKLOADS["rope_quant_tiny"].make()
    g = _cuda(d)
    y, q, s = fq.rmsnorm_rope_quant(g["x"], g["w"], g["cos"], g["sin"])
    y_ref, q_ref, s_ref = orc.rmsnorm_rope_quant(d["x"], d["w"], d["cos"], d["sin"])
    assert_rope_close(y, y_ref, orc.rmsnorm_fwd(d["x"], d["w"]), d["cos"], d["sin"])
    q_own, s_own = orc.quant_rows(y.cpu())
    assert_own_quantiser(q, s, q_own, s_own)
    assert_codes_close(q, q_ref)
    assert scale_rows_by_own_y(s, s_ref) == 0
    assert_scale_close(s, s_ref)
