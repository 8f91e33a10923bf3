"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every entry point that
include/fq.h declares, and rejects invalid arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest
import torch

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from fp8_quant_memory_gb300 import _capi, build

    try:
        build.build()
    except RuntimeError as e:  # no nvcc on this machine
        pytest.skip(str(e))
    return _capi.load()


def _declared():
    with open(os.path.join(ROOT, "include", "fq.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("fq_rmsnorm_fwd", "fq_rmsnorm_bwd", "fq_rmsnorm_rope", "fq_rmsnorm_rope_quant",
              "fq_qk_norm_rope_quant", "fq_rmsnorm_bwd_workspace_bytes", "fq_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from fp8_quant_memory_gb300 import _capi

    for name in _declared():
        assert hasattr(lib, name), name
        assert name in _capi.SIGNATURES, f"binding has no signature for {name}"


def test_version(lib):
    assert lib.fq_version() >= 1


NULL = None


def _rc(lib, name, *args):
    rc = getattr(lib, name)(*args)
    return rc, lib.fq_last_error().decode()


def test_null_pointers_rejected(lib):
    p = ctypes.c_void_p(16)
    rc, msg = _rc(lib, "fq_rmsnorm_fwd", NULL, p, p, 4, 8, 0, 1e-6, NULL)
    assert rc == 1 and "null" in msg
    rc, _ = _rc(lib, "fq_rmsnorm_rope_quant", p, p, p, p, NULL, p, NULL, 4, 8, 4, 0, 0, 1e-6, 448.0, NULL)
    assert rc == 1
    rc, _ = _rc(lib, "fq_qk_norm_rope_quant", p, 1024, p, NULL, p, p, p, p, 2, 4, 4, 128, 128, 0, 2, 1e-6,
                448.0, NULL)
    assert rc == 1


def test_bad_dtypes_rejected(lib):
    p = ctypes.c_void_p(16)
    rc, msg = _rc(lib, "fq_rmsnorm_fwd", p, p, p, 4, 8, 2, 1e-6, NULL)  # fp32 storage not accepted
    assert rc == 2 and "dtype" in msg
    rc, _ = _rc(lib, "fq_rmsnorm_rope", p, p, p, p, p, 4, 64, 32, 0, 7, 1e-6, NULL)
    assert rc == 2


def test_shape_rules_rejected(lib):
    p = ctypes.c_void_p(16)
    # odd rope_dim, rope_dim > N
    assert _rc(lib, "fq_rmsnorm_rope", p, p, p, p, p, 4, 64, 31, 0, 0, 1e-6, NULL)[0] == 1
    assert _rc(lib, "fq_rmsnorm_rope", p, p, p, p, p, 4, 64, 66, 0, 0, 1e-6, NULL)[0] == 1
    # N < 1, M < 0
    assert _rc(lib, "fq_rmsnorm_fwd", p, p, p, 4, 0, 0, 1e-6, NULL)[0] == 1
    assert _rc(lib, "fq_rmsnorm_fwd", p, p, p, -1, 8, 0, 1e-6, NULL)[0] == 1
    # fp8_max outside (0, 448]; eps negative or NaN
    assert _rc(lib, "fq_rmsnorm_rope_quant", p, p, p, p, NULL, p, p, 4, 8, 4, 0, 0, 1e-6, 449.0, NULL)[0] == 1
    assert _rc(lib, "fq_rmsnorm_rope_quant", p, p, p, p, NULL, p, p, 4, 8, 4, 0, 0, 1e-6, 0.0, NULL)[0] == 1
    assert _rc(lib, "fq_rmsnorm_fwd", p, p, p, 4, 8, 0, -1.0, NULL)[0] == 1
    assert _rc(lib, "fq_rmsnorm_fwd", p, p, p, 4, 8, 0, float("nan"), NULL)[0] == 1
    # token stride shorter than the heads, no heads at all
    rc, msg = _rc(lib, "fq_qk_norm_rope_quant", p, 1000, p, p, p, p, p, p, 2, 4, 4, 128, 128, 0, 2, 1e-6,
                  448.0, NULL)
    assert rc == 1 and "token_stride" in msg
    assert _rc(lib, "fq_qk_norm_rope_quant", p, 0, p, p, p, p, p, p, 2, 0, 0, 128, 128, 0, 2, 1e-6, 448.0,
               NULL)[0] == 1
    # rows that overflow 32-bit row indexing
    assert _rc(lib, "fq_qk_norm_rope_quant", p, 40 * 128, p, p, p, p, p, p, 2 ** 30, 32, 8, 128, 128, 0, 2,
               1e-6, 448.0, NULL)[0] == 1


def test_saved_rstd_rules(lib):
    p = ctypes.c_void_p(16)
    rc, msg = _rc(lib, "fq_rmsnorm_bwd_rstd", p, p, p, NULL, p, p, NULL, p, 1 << 20, 8, 64, 0, NULL)
    assert rc == 1 and "rstd" in msg
    assert _rc(lib, "fq_rmsnorm_fwd_rstd", p, p, NULL, p, 4, 8, 0, 1e-6, NULL)[0] == 1  # null y
    assert _rc(lib, "fq_rmsnorm_fwd_rstd", p, p, p, NULL, 0, 8, 0, 1e-6, NULL)[0] == 0  # empty


def test_group_size_rules_rejected(lib):
    """Group-wise scales: group_size must be >= 1 and divide N; checked on the host."""
    p = ctypes.c_void_p(16)
    f = "fq_rmsnorm_rope_quant_groups"
    rc, msg = _rc(lib, f, p, p, p, p, NULL, p, p, 4, 512, 64, 96, 0, 0, 1e-6, 448.0, NULL)
    assert rc == 1 and "group_size" in msg
    assert _rc(lib, f, p, p, p, p, NULL, p, p, 4, 512, 64, 0, 0, 0, 1e-6, 448.0, NULL)[0] == 1
    assert _rc(lib, f, p, p, p, p, NULL, p, p, 4, 512, 64, -8, 0, 0, 1e-6, 448.0, NULL)[0] == 1
    assert _rc(lib, f, p, p, p, p, NULL, NULL, p, 4, 512, 64, 128, 0, 0, 1e-6, 448.0, NULL)[0] == 1  # null q
    assert _rc(lib, f, p, p, p, p, NULL, p, p, 0, 512, 64, 128, 0, 0, 1e-6, 448.0, NULL)[0] == 0     # empty


def test_empty_batches_are_noops_without_cuda(lib):
    p = ctypes.c_void_p(16)
    assert _rc(lib, "fq_rmsnorm_fwd", p, p, p, 0, 8, 0, 1e-6, NULL)[0] == 0
    assert _rc(lib, "fq_qk_norm_rope_quant", p, 512, p, p, p, p, p, p, 0, 2, 2, 128, 128, 0, 2, 1e-6, 448.0,
               NULL)[0] == 0


def test_bwd_workspace_rules(lib):
    ws = lib.fq_rmsnorm_bwd_workspace_bytes
    assert ws(0, 4096) == 0
    assert ws(8192, 4096) == 256 * 4096 * 4  # 256 chunks of 32 rows
    assert ws(100, 64) == 100 * 64 * 4       # one row per chunk when M <= 256
    assert ws(257, 16) == 129 * 16 * 4       # 2 rows per chunk
    p = ctypes.c_void_p(16)
    rc, msg = _rc(lib, "fq_rmsnorm_bwd", p, p, p, p, p, NULL, p, 100, 8192, 4096, 0, 1e-6, NULL)
    assert rc == 1 and "workspace" in msg
    rc, msg = _rc(lib, "fq_rmsnorm_bwd", p, p, p, p, p, NULL, ctypes.c_void_p(24), 2 ** 24, 8192, 4096, 0,
                  1e-6, NULL)
    assert rc == 1 and "aligned" in msg


def test_binding_rejects_host_tensors():
    import fp8_quant_memory_gb300 as fq

    x = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fq.rmsnorm_fwd(x, torch.ones(8, dtype=torch.bfloat16))


def test_stream_floor_rules(lib):
    p, odd = ctypes.c_void_p(16), ctypes.c_void_p(24)
    assert _rc(lib, "fq_stream_floor", p, p, 0, NULL)[0] == 0          # nothing to stream: no-op
    rc, msg = _rc(lib, "fq_stream_floor", NULL, p, 4, NULL)
    assert rc == 1 and "null" in msg
    assert _rc(lib, "fq_stream_floor", p, p, -1, NULL)[0] == 1
    rc, msg = _rc(lib, "fq_stream_floor", odd, p, 4, NULL)             # input not 16-byte aligned
    assert rc == 1 and "aligned" in msg
    assert _rc(lib, "fq_stream_floor", p, ctypes.c_void_p(20), 4, NULL)[0] == 1


def test_layernorm_rules(lib):
    p = ctypes.c_void_p(16)
    assert _rc(lib, "fq_layernorm_fwd", p, p, NULL, p, 0, 64, 0, 1e-5, NULL)[0] == 0    # M = 0: no-op
    rc, msg = _rc(lib, "fq_layernorm_fwd", p, NULL, NULL, p, 4, 64, 0, 1e-5, NULL)      # no gain
    assert rc == 1 and "null" in msg
    assert _rc(lib, "fq_layernorm_fwd", p, p, NULL, p, 4, 0, 0, 1e-5, NULL)[0] == 1     # N = 0
    assert _rc(lib, "fq_layernorm_fwd", p, p, NULL, p, 4, 64, 2, 1e-5, NULL)[0] == 2    # fp32 storage
    assert _rc(lib, "fq_layernorm_fwd", p, p, NULL, p, 4, 64, 0, -1.0, NULL)[0] == 1    # eps < 0


def test_prologue_blocks_rules(lib):
    p = ctypes.c_void_p(16)
    args = (p, 1024, p, p, p, p, p, p, 2, 4, 4, 128, 128)
    for rpb in (0, 129):
        rc, msg = _rc(lib, "fq_qk_norm_rope_quant_blocks", *args, rpb, 0, 2, 1e-6, 448.0, NULL)
        assert rc == 1 and "rows_per_block" in msg
    assert _rc(lib, "fq_qk_norm_rope_quant_blocks", p, 1024, p, p, p, p, p, p, 0, 4, 4, 128, 128, 8, 0, 2, 1e-6,
               448.0, NULL)[0] == 0                                                        # T = 0: no-op


def test_bounded_wait_limit_rules(lib):
    for ms in (0, 10001):
        rc, msg = _rc(lib, "fq_check_bounded_wait", ms, NULL)
        assert rc == 1 and "limit_ms" in msg


def test_strict_mode_toggles_without_a_device(lib):
    """fq_set_strict only sets a flag (the synchronisation happens in later compute calls)."""
    prev = lib.fq_set_strict(1)
    try:
        assert lib.fq_set_strict(0) == 1
        assert lib.fq_set_strict(1) == 0
    finally:
        lib.fq_set_strict(prev)


def test_version_counts_the_strict_mode_entry_point(lib):
    assert lib.fq_version() >= 2
