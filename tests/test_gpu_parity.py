"""GPU parity: every libfq entry point against the oracle on the same seeded inputs, at sizes the
oracle finishes in seconds that span many CTAs and a ragged tail, plus edge cases (one row, an
empty batch, odd widths and misaligned views that take the scalar kernel, a token stride, a
non-default fp8_max, partial rope). Tolerances: tests/parity.py.
"""
import pytest
import torch

import fp8_quant_memory_gb300 as fq
from fp8_quant_memory_gb300 import workloads as wl
from parity import (assert_own_quantiser, assert_codes_close, assert_dw_close, assert_rope_close, assert_scale_close,
                    assert_storage_close, assert_within_one_ulp, scale_rows_by_own_y)

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def cuda(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def misalign(t: torch.Tensor) -> torch.Tensor:
    """Same values at an address that is 2 bytes past a 16-byte boundary (forces the scalar path)."""
    flat = torch.empty(t.numel() + 8, dtype=t.dtype, device=t.device)
    view = flat[1: 1 + t.numel()].view(t.shape)
    view.copy_(t)
    return view


# ----------------------------------------------------------------------------------- prologue
PROLOGUE_CASES = [
    # T, Hq, Hk, D, R, dtype, table, std, stride_extra, fp8_max
    (37, 32, 8, 128, 128, "bf16", "fp32", 2.0, 0, 448.0),
    (1, 32, 8, 128, 128, "bf16", "fp32", 2.0, 0, 448.0),
    (129, 4, 2, 128, 128, "fp16", "fp32", 1.0, 0, 448.0),
    (50, 6, 2, 128, 128, "bf16", "bf16", 1.0, 0, 448.0),
    (33, 3, 1, 128, 128, "bf16", "fp32", 1.0, 3 * 128, 448.0),   # q/k slice of a QKV row
    (17, 8, 0, 64, 64, "bf16", "fp32", 1.0, 0, 448.0),           # q only, D = 64
    (21, 0, 4, 128, 64, "bf16", "fp32", 1.0, 0, 448.0),          # k only, partial rope
    (19, 5, 3, 256, 128, "fp16", "fp16", 1.0, 0, 448.0),         # D = 256
    (23, 4, 4, 128, 128, "bf16", "fp32", 1.0, 0, 240.0),         # fp8_max < 448
    (13, 3, 2, 96, 40, "bf16", "fp32", 1.0, 0, 448.0),           # rope_dim not a multiple of 16
    (11, 2, 2, 100, 50, "bf16", "bf16", 1.0, 0, 448.0),          # odd-ish width: scalar path
    (9, 2, 1, 128, 0, "bf16", "fp32", 1.0, 0, 448.0),            # no rotation
    (7, 40, 8, 128, 128, "bf16", "fp16", 1.0, 0, 448.0),         # table dtype != storage dtype
    (29, 16, 8, 128, 128, "bf16", "fp32", 1.0, 0, 240.0),        # head counts multiples of 8, fp8_max < 448
    (31, 8, 8, 128, 128, "fp16", "fp16", 1.0, 0, 448.0),         # head counts multiples of 8, fp16 tables
]


def _run_prologue(orc, case, seed=100, force_scalar=False):
    T, Hq, Hk, D, R, dt, tdt, std, extra, fmax = case
    H = Hq + Hk
    ts = None if extra == 0 else H * D + extra
    d = wl.qk_inputs(T, Hq, Hk, D, dt, tdt, seed=seed, std=std, rope_dim=R, token_stride=ts)
    q_ref, s_ref = orc.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], Hq, Hk,
                                          fp8_max=fmax, rope_dim=R)
    g = cuda(d)
    qk = misalign(g["qk"]) if force_scalar else g["qk"]
    q, s = fq.qk_norm_rope_quant(qk, g["wq"], g["wk"], g["cos"], g["sin"], Hq, Hk, fp8_max=fmax, rope_dim=R)
    torch.cuda.synchronize()
    assert_scale_close(s, s_ref)
    assert_codes_close(q, q_ref)


@pytest.mark.parametrize("case", PROLOGUE_CASES, ids=lambda c: "T%d-%d+%d-D%d-R%d-%s-%s-x%d-m%g" % (
    c[0], c[1], c[2], c[3], c[4], c[5], c[6], c[8], c[9]))
def test_prologue_parity(orc, cuda_ok, case):
    _run_prologue(orc, case)


@pytest.mark.parametrize("case", PROLOGUE_CASES[:4], ids=lambda c: "T%d-%d+%d-%s" % (c[0], c[1], c[2], c[5]))
def test_prologue_parity_scalar_path(orc, cuda_ok, case):
    _run_prologue(orc, case, seed=101, force_scalar=True)


def test_prologue_empty_batch(cuda_ok):
    d = cuda(wl.qk_inputs(1, 2, 2, 128, seed=1))
    q, s = fq.qk_norm_rope_quant(d["qk"][:0], d["wq"], d["wk"], d["cos"][:0], d["sin"][:0], 2, 2)
    torch.cuda.synchronize()
    assert q.shape == (0, 4, 128) and s.shape == (0, 4)


def test_prologue_outliers_and_huge_positions(orc, cuda_ok):
    """Config-5-like statistics (1% outliers x50, positions up to 131072, theta 1e6), small T."""
    d = wl.qk_inputs(64, 16, 4, 128, "bf16", "fp32", seed=102, std=1.0, theta=1e6, positions="uniform",
                     outlier_frac=0.01)
    q_ref, s_ref = orc.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], 16, 4)
    g = cuda(d)
    q, s = fq.qk_norm_rope_quant(g["qk"], g["wq"], g["wk"], g["cos"], g["sin"], 16, 4)
    assert_scale_close(s, s_ref)
    assert_codes_close(q, q_ref)


def test_prologue_zero_rows(orc, cuda_ok):
    """All-zero rows: scale = 1e-4/448 and every code decodes to zero. The rotation can give -0
    (0*c - 0*s with c < 0 < s), which e4m3fn encodes as 0x80, so the sign bit is not checked."""
    d = wl.qk_inputs(4, 2, 2, 128, seed=103)
    d["qk"][1:3] = 0
    q_ref, s_ref = orc.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], 2, 2)
    g = cuda(d)
    q, s = fq.qk_norm_rope_quant(g["qk"], g["wq"], g["wk"], g["cos"], g["sin"], 2, 2)
    assert int((q.cpu()[1:3] & 0x7F).max()) == 0
    assert torch.equal(s.cpu()[1:3], s_ref[1:3])
    assert_codes_close(q, q_ref)


# ----------------------------------------------------------------------------------- rmsnorm_rope_quant
ROPE_QUANT_CASES = [
    # M, N, R, dtype, table
    (256, 512, 64, "bf16", "bf16"),    # the tiny workload
    (1, 512, 64, "bf16", "bf16"),
    (37, 192, 64, "fp16", "fp16"),
    (300, 128, 128, "bf16", "fp32"),
    (64, 4096, 128, "fp16", "fp16"),   # the fusion page's own demo width
    (45, 1024, 256, "bf16", "bf16"),
    (33, 100, 20, "bf16", "bf16"),     # scalar path
    (29, 256, 0, "bf16", "bf16"),      # no rotation
    (31, 512, 64, "bf16", "fp16"),     # mixed table dtype: scalar path
]


@pytest.mark.parametrize("want_y", [True, False])
@pytest.mark.parametrize("case", ROPE_QUANT_CASES, ids=lambda c: "M%d-N%d-R%d-%s-%s" % c)
def test_rmsnorm_rope_quant_parity(orc, cuda_ok, case, want_y):
    M, N, R, dt, tdt = case
    d = wl.rows_inputs(M, N, R, dt, tdt, seed=200 + M)
    y_ref, q_ref, s_ref = orc.rmsnorm_rope_quant(d["x"], d["w"], d["cos"], d["sin"])
    g = cuda(d)
    y, q, s = fq.rmsnorm_rope_quant(g["x"], g["w"], g["cos"], g["sin"], want_y=True)
    torch.cuda.synchronize()
    assert_rope_close(y, y_ref, orc.rmsnorm_fwd(d["x"], d["w"]), d["cos"], d["sin"])
    # The scales are the quantiser applied to the kernel's own y exactly, the codes under the code rule.
    q_own, s_own = orc.quant_rows(y.cpu())
    assert_own_quantiser(q, s, q_own, s_own)
    assert_codes_close(q, q_ref)
    # Scales within 1e-5 of the oracle's, except rows accepted by the own-y rule above (a bf16 flip
    # of the amax element); none on the tiny workload, and rare elsewhere.
    n_own = scale_rows_by_own_y(s, s_ref)
    if (M, N, R, dt, tdt) == (256, 512, 64, "bf16", "bf16"):
        assert n_own == 0
        assert_scale_close(s, s_ref)
    assert n_own <= max(1, M // 1000), f"{n_own} of {M} rows accepted only by the own-y rule"
    if not want_y:
        _, q2, s2 = fq.rmsnorm_rope_quant(g["x"], g["w"], g["cos"], g["sin"], want_y=False)
        assert torch.equal(q2, q) and torch.equal(s2, s)


def test_rmsnorm_rope_quant_scalar_path_matches(orc, cuda_ok):
    d = wl.rows_inputs(77, 512, 64, "bf16", "bf16", seed=250)
    y_ref, q_ref, _ = orc.rmsnorm_rope_quant(d["x"], d["w"], d["cos"], d["sin"])
    g = cuda(d)
    y, q, s = fq.rmsnorm_rope_quant(misalign(g["x"]), g["w"], g["cos"], g["sin"])
    assert_rope_close(y, y_ref, orc.rmsnorm_fwd(d["x"], d["w"]), d["cos"], d["sin"])
    q_own, s_own = orc.quant_rows(y.cpu())
    assert_own_quantiser(q, s, q_own, s_own)


# ----------------------------------------------------------------------------------- group-wise scales
GROUP_CASES = [
    # M, N, R, group_size, dtype, table
    (256, 512, 64, 128, "bf16", "bf16"),   # the tiny workload, 4 groups (the last spans head and tail)
    (300, 512, 64, 64, "fp16", "fp32"),
    (100, 192, 64, 32, "bf16", "bf16"),    # groups inside the tail-lo / tail-hi halves
    (77, 4096, 128, 128, "bf16", "bf16"),  # 32 groups on a wide row
    (50, 1024, 0, 8, "bf16", "bf16"),      # the smallest vector group, no rotation
    (9, 2048, 64, 8, "fp16", "fp16"),      # 256 groups per row
    (33, 96, 32, 12, "bf16", "bf16"),      # group not a multiple of 8: scalar kernel
    (40, 100, 50, 25, "bf16", "fp32"),     # odd width: scalar kernel
    (5, 64, 16, 1, "bf16", "bf16"),        # one column per group: scalar kernel
]


@pytest.mark.parametrize("case", GROUP_CASES, ids=lambda c: "M%d-N%d-R%d-g%d-%s-%s" % c)
def test_rmsnorm_rope_quant_groups_parity(orc, cuda_ok, case):
    M, N, R, gs, dt, tdt = case
    d = wl.rows_inputs(M, N, R, dt, tdt, seed=260 + M)
    y_ref, q_ref, s_ref = orc.rmsnorm_rope_quant_groups(d["x"], d["w"], d["cos"], d["sin"], gs)
    g = cuda(d)
    y, q, s = fq.rmsnorm_rope_quant_groups(g["x"], g["w"], g["cos"], g["sin"], gs)
    torch.cuda.synchronize()
    assert s.shape == (M, N // gs)
    assert_rope_close(y, y_ref, orc.rmsnorm_fwd(d["x"], d["w"]), d["cos"], d["sin"])
    # the group-wise quantiser applied to the kernel's own y: scales exactly, codes under the code rule
    q_own, s_own = orc.quant_groups(y.cpu(), gs)
    assert_own_quantiser(q, s, q_own, s_own)
    assert_codes_close(q, q_ref)
    n_own = scale_rows_by_own_y(s, s_ref)
    assert n_own <= max(1, s.numel() // 1000), f"{n_own} of {s.numel()} group scales accepted only by the own-y rule"
    _, q2, s2 = fq.rmsnorm_rope_quant_groups(g["x"], g["w"], g["cos"], g["sin"], gs, want_y=False)
    assert torch.equal(q2, q) and torch.equal(s2, s)
    assert fq.device_status(clear=True) == 0


def test_rmsnorm_rope_quant_groups_one_group_is_per_row(cuda_ok):
    """group_size = N is the per-row entry point, bit for bit."""
    g = cuda(wl.rows_inputs(128, 512, 64, "bf16", "bf16", seed=290))
    y1, q1, s1 = fq.rmsnorm_rope_quant(g["x"], g["w"], g["cos"], g["sin"])
    y2, q2, s2 = fq.rmsnorm_rope_quant_groups(g["x"], g["w"], g["cos"], g["sin"], 512)
    assert torch.equal(y1, y2) and torch.equal(q1, q2) and torch.equal(s1, s2[:, 0])


def test_rmsnorm_rope_quant_groups_scalar_path_matches(orc, cuda_ok):
    """A vector-eligible shape at a misaligned address takes the scalar kernel: same rules."""
    d = wl.rows_inputs(61, 512, 64, "bf16", "bf16", seed=291)
    y_ref, q_ref, _ = orc.rmsnorm_rope_quant_groups(d["x"], d["w"], d["cos"], d["sin"], 128)
    g = cuda(d)
    y, q, s = fq.rmsnorm_rope_quant_groups(misalign(g["x"]), g["w"], g["cos"], g["sin"], 128)
    assert_rope_close(y, y_ref, orc.rmsnorm_fwd(d["x"], d["w"]), d["cos"], d["sin"])
    q_own, s_own = orc.quant_groups(y.cpu(), 128)
    assert_own_quantiser(q, s, q_own, s_own)


# ----------------------------------------------------------------------------------- wide quantising rows
WIDE_QUANT_CASES = [
    # M, N, R, group_size (None: one scale per row), dtype, table, write y
    (4096, 4096, 128, None, "bf16", "bf16", False),  # the Ch.13 ledger's fused workload
    (4096, 4096, 128, 128, "bf16", "bf16", True),
    (4099, 1024, 64, 8, "fp16", "fp32", True),        # 128 groups per row, ragged last stage
    (4100, 2048, 0, None, "bf16", "bf16", True),      # no rotation
    (4097, 1536, 256, 512, "bf16", "fp32", False),    # groups spanning head and tail
    (4096, 3072, 128, 1024, "bf16", "fp32", True),    # a group spans four 32-vector slots
    (4098, 4096, 256, 512, "fp16", "fp32", False),    # every last-slot lane rotary; groups of two slots
    (4096, 2048, 32, 2048, "bf16", "bf16", True),     # one group per row through the group entry point
    (4101, 3072, 16, None, "fp16", "fp16", False),    # one rotary pair block per half
    (4102, 1024, 64, 128, "fp16", "fp32", True),      # groups of 128, four slots per lane
    (4096, 2048, 128, 128, "bf16", "fp32", False),    # groups of 128, eight slots per lane
    (4097, 4096, 64, 64, "bf16", "bf16", False),      # groups of 64 on the widest rows
    (4099, 3072, 128, 128, "bf16", "bf16", True),     # groups of 128, twelve slots per lane (3 blocks)
    (4096, 4096, 128, 4096, "bf16", "fp32", True),    # one group per 4096-wide row: the per-row kernel
]


@pytest.mark.parametrize("kernel", ["tma", "staged", "generic"])
@pytest.mark.parametrize("case", WIDE_QUANT_CASES, ids=lambda c: "M%d-N%d-R%d-g%s-%s-%s-y%d" % c)
def test_wide_rows_quant_stream_kernel(orc, cuda_ok, monkeypatch, case, kernel):
    """RMSNorm + RoPE + FP8 on >= 4096 rows of >= 1024 elements (the TMA-fed register-resident kernel
    where the width, rope_dim and group size allow it, the TMA-fed shared-memory kernel, and the
    generic kernel on the same inputs): y against the oracle, scales exactly and codes under the code
    rule against the quantiser of the kernel's own y."""
    _rows_kernel(monkeypatch, kernel)
    M, N, R, gs, dt, tdt, want_y = case
    d = wl.rows_inputs(M, N, R, dt, tdt, seed=970 + M)
    g = cuda(d)
    if gs is None:
        y_ref, q_ref, s_ref = orc.rmsnorm_rope_quant(d["x"], d["w"], d["cos"], d["sin"])
        y, q, sc = fq.rmsnorm_rope_quant(g["x"], g["w"], g["cos"], g["sin"], want_y=True)
        q_own, s_own = orc.quant_rows(y.cpu())
    else:
        y_ref, q_ref, s_ref = orc.rmsnorm_rope_quant_groups(d["x"], d["w"], d["cos"], d["sin"], gs)
        y, q, sc = fq.rmsnorm_rope_quant_groups(g["x"], g["w"], g["cos"], g["sin"], gs, want_y=True)
        q_own, s_own = orc.quant_groups(y.cpu(), gs)
    torch.cuda.synchronize()
    assert_rope_close(y, y_ref, orc.rmsnorm_fwd(d["x"], d["w"]), d["cos"], d["sin"])
    assert_own_quantiser(q, sc, q_own, s_own)
    assert_codes_close(q, q_ref)
    n_own = scale_rows_by_own_y(sc, s_ref)
    assert n_own <= max(1, sc.numel() // 1000), f"{n_own} of {sc.numel()} scales accepted only by the own-y rule"
    if gs == N:  # a whole-row group is the per-row entry point, bit for bit
        y1, q1, s1 = fq.rmsnorm_rope_quant(g["x"], g["w"], g["cos"], g["sin"], want_y=True)
        assert torch.equal(y1, y) and torch.equal(q1, q) and torch.equal(s1, sc[:, 0])
    if not want_y:
        if gs is None:
            _, q2, s2 = fq.rmsnorm_rope_quant(g["x"], g["w"], g["cos"], g["sin"], want_y=False)
        else:
            _, q2, s2 = fq.rmsnorm_rope_quant_groups(g["x"], g["w"], g["cos"], g["sin"], gs, want_y=False)
        assert torch.equal(q2, q) and torch.equal(s2, sc)
    assert fq.device_status(clear=True) == 0


@pytest.mark.parametrize("path", ["vector", "wide_stream", "scalar", "groups", "prologue_tma", "prologue_generic"])
def test_negative_zero_inputs_give_negative_zero_codes(orc, cuda_ok, monkeypatch, path):
    """x = -0.0 normalises (and, with angle-free columns, quantises) to -0: the definition's y / scale
    keeps the sign of zero and e4m3fn codes it 0x80. Planted -0.0 (and +0.0) entries on every path."""
    monkeypatch.delenv("FQ_PROLOGUE_KERNEL", raising=False)
    monkeypatch.delenv("FQ_ROWS_KERNEL", raising=False)
    if path.startswith("prologue"):
        if path == "prologue_generic":
            monkeypatch.setenv("FQ_PROLOGUE_KERNEL", "generic")
        d = wl.qk_inputs(64, 4, 2, 128, "bf16", "fp32", seed=995, std=1.0)
        d["qk"][3, 1, 5] = -0.0
        d["qk"][7, 4, 100] = -0.0
        d["qk"][9, 0, 17] = 0.0
        q_ref, s_ref = orc.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], 4, 2)
        g = cuda(d)
        q, s = fq.qk_norm_rope_quant(g["qk"], g["wq"], g["wk"], g["cos"], g["sin"], 4, 2)
        torch.cuda.synchronize()
        assert_codes_close(q, q_ref)
        assert_scale_close(s, s_ref)
        return
    M, N, R = (4096, 1024, 64) if path == "wide_stream" else (64, 512, 64)
    d = wl.rows_inputs(M, N, R, "bf16", "bf16", seed=996)
    planted = [(1, 7), (2, 300), (5, 0), (M - 1, N - R - 1)]  # head columns: y = -0 exactly
    for (i, j) in planted:
        d["x"][i, j] = -0.0
    d["x"][3, 11] = 0.0
    g = cuda(d)
    x = misalign(g["x"]) if path == "scalar" else g["x"]
    if path == "groups":
        y, q, s = fq.rmsnorm_rope_quant_groups(x, g["w"], g["cos"], g["sin"], 128)
        q_own, s_own = orc.quant_groups(y.cpu(), 128)
    else:
        y, q, s = fq.rmsnorm_rope_quant(x, g["w"], g["cos"], g["sin"])
        q_own, s_own = orc.quant_rows(y.cpu())
    torch.cuda.synchronize()
    qc = q.cpu()
    for (i, j) in planted:
        assert torch.signbit(y.cpu()[i, j]) and float(y.cpu()[i, j]) == 0.0
        assert int(qc[i, j]) == 0x80
    assert int(qc[3, 11]) == 0x00
    assert_own_quantiser(qc, s, q_own, s_own)


# ----------------------------------------------------------------------------------- rmsnorm_rope
@pytest.mark.parametrize("case", [(4096, 192, 64, "fp16", "fp16", 32), (100, 192, 64, "bf16", "fp32", 1),
                                  (64, 256, 32, "bf16", "bf16", 1), (10, 70, 14, "fp16", "fp16", 1)],
                         ids=lambda c: "M%d-N%d-R%d-%s-%s-h%d" % c)
def test_rmsnorm_rope_parity(orc, cuda_ok, case):
    M, N, R, dt, tdt, hpt = case
    d = wl.rows_inputs(M, N, R, dt, tdt, seed=300 + M, heads_per_token=hpt)
    y_ref = orc.rmsnorm_rope(d["x"], d["w"], d["cos"], d["sin"])
    g = cuda(d)
    y = fq.rmsnorm_rope(g["x"], g["w"], g["cos"], g["sin"])
    assert_rope_close(y, y_ref, orc.rmsnorm_fwd(d["x"], d["w"]), d["cos"], d["sin"])


# ----------------------------------------------------------------------------------- rmsnorm fwd
@pytest.mark.parametrize("case", [(64, 4096, "bf16"), (513, 128, "bf16"), (33, 2048, "fp16"), (1, 8, "bf16"),
                                  (17, 100, "bf16"), (5, 5000, "fp16")], ids=lambda c: "M%d-N%d-%s" % c)
def test_rmsnorm_fwd_parity(orc, cuda_ok, case):
    M, N, dt = case
    d = wl.rmsnorm_inputs(M, N, dt, seed=400 + M)
    y_ref = orc.rmsnorm_fwd(d["x"], d["w"])
    g = cuda(d)
    y = fq.rmsnorm_fwd(g["x"], g["w"])
    assert_storage_close(y, y_ref)


def test_rmsnorm_fwd_empty(cuda_ok):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    y = fq.rmsnorm_fwd(x, torch.ones(64, dtype=torch.bfloat16, device="cuda"))
    assert y.shape == (0, 64)


# ----------------------------------------------------------------------------------- backward
@pytest.mark.parametrize("case", [(257, 4096, "bf16"), (300, 128, "bf16"), (70, 1024, "fp16"),
                                  (1, 512, "bf16"), (41, 100, "bf16"), (9, 8192, "bf16"), (600, 2048, "fp16")],
                         ids=lambda c: "M%d-N%d-%s" % c)
def test_rmsnorm_bwd_parity(orc, cuda_ok, case):
    M, N, dt = case
    d = wl.rmsnorm_inputs(M, N, dt, seed=500 + M)
    dx_ref, dw_ref, dw32_ref = orc.rmsnorm_bwd(d["x"], d["w"], d["g"])
    g = cuda(d)
    dx, dw, dw32 = fq.rmsnorm_bwd(g["x"], g["w"], g["g"])
    assert_storage_close(dx, dx_ref, "dx")
    assert_dw_close(dw32, dw32_ref)
    assert_within_one_ulp(dw, dw_ref)
    assert torch.equal(dw.cpu(), dw32.cpu().to(dw.dtype))


@pytest.mark.parametrize("kernel", ["stream", "generic"])
@pytest.mark.parametrize("case", [(1000, 1536, "bf16"), (513, 4096, "fp16"), (300, 2056, "bf16")],
                         ids=lambda c: "M%d-N%d-%s" % c)
def test_rmsnorm_bwd_stream_kernel(orc, cuda_ok, monkeypatch, case, kernel):
    """The TMA-fed stage 1 (rows of 1032..4096 elements) and the global-load stage 1 against the
    oracle; idle column threads (N not a multiple of 2048) and fp16 included."""
    M, N, dt = case
    if kernel == "generic":
        monkeypatch.setenv("FQ_BWD_KERNEL", "generic")
    else:
        monkeypatch.delenv("FQ_BWD_KERNEL", raising=False)
    d = wl.rmsnorm_inputs(M, N, dt, seed=580 + M)
    dx_ref, dw_ref, dw32_ref = orc.rmsnorm_bwd(d["x"], d["w"], d["g"])
    g = cuda(d)
    dx, dw, dw32 = fq.rmsnorm_bwd(g["x"], g["w"], g["g"])
    assert_storage_close(dx, dx_ref, "dx")
    assert_dw_close(dw32, dw32_ref)
    assert_within_one_ulp(dw, dw_ref)
    assert fq.device_status(clear=True) == 0


def test_rmsnorm_bwd_stream_matches_generic_bitwise(cuda_ok, monkeypatch):
    """Both stage-1 kernels give each thread the same columns and add in the same order: dx and the
    fp32 dw sums agree bit for bit."""
    d = cuda(wl.rmsnorm_inputs(777, 4096, "bf16", seed=590))
    monkeypatch.delenv("FQ_BWD_KERNEL", raising=False)
    a = fq.rmsnorm_bwd(d["x"], d["w"], d["g"])
    monkeypatch.setenv("FQ_BWD_KERNEL", "generic")
    b = fq.rmsnorm_bwd(d["x"], d["w"], d["g"])
    for u, v in zip(a, b):
        assert torch.equal(u, v)


# saved rstd: shapes that reach every forward kernel (generic narrow and wide, TMA narrow and wide,
# scalar) and every backward stage 1 (TMA-fed, global-load, scalar)
RSTD_CASES = [
    # M, N, dtype, misalign
    (300, 256, "bf16", False),     # generic narrow rows
    (129, 2048, "fp16", False),    # generic wide rows
    (4100, 512, "bf16", False),    # TMA narrow rows
    (4097, 4096, "bf16", False),   # TMA wide rows (two warps per row); TMA-fed backward
    (4099, 1536, "fp16", False),   # TMA wide rows, one warp per row
    (77, 1024, "bf16", False),     # global-load backward
    (45, 100, "bf16", False),      # odd width: scalar forward and backward
    (60, 512, "bf16", True),       # misaligned: scalar
]


@pytest.mark.parametrize("case", RSTD_CASES, ids=lambda c: "M%d-N%d-%s-mis%d" % c)
def test_rmsnorm_saved_rstd(orc, cuda_ok, case):
    M, N, dt, mis = case
    d = wl.rmsnorm_inputs(M, N, dt, seed=700 + M)
    y_ref, r_ref = orc.rmsnorm_fwd_rstd(d["x"], d["w"])
    g = cuda(d)
    x = misalign(g["x"]) if mis else g["x"]
    y, rstd = fq.rmsnorm_fwd_rstd(x, g["w"])
    torch.cuda.synchronize()
    assert_storage_close(y, y_ref)
    rel = ((rstd.cpu().double() - r_ref.double()).abs() / r_ref.double()).max().item()
    assert rel <= 1e-6, rel  # rstd differs from the oracle's only by the fp32 order of the sum of squares
    assert torch.equal(y, fq.rmsnorm_fwd(x, g["w"]))  # the rstd output does not change y
    # backward with the saved rstd: against the oracle given the same rstd, and against the recomputing one
    dx, dw, dw32 = fq.rmsnorm_bwd_rstd(x, g["w"], g["g"], rstd)
    dx_o, dw_o, dw32_o = orc.rmsnorm_bwd_rstd(d["x"], d["w"], d["g"], rstd.cpu())
    assert_storage_close(dx, dx_o, "dx")
    assert_dw_close(dw32, dw32_o)
    assert_within_one_ulp(dw, dw_o)
    dx_r, _, dw32_r = orc.rmsnorm_bwd(d["x"], d["w"], d["g"])
    assert_storage_close(dx, dx_r, "dx")
    assert_dw_close(dw32, dw32_r)
    assert fq.device_status(clear=True) == 0


def test_rmsnorm_autograd_save_rstd(cuda_ok):
    d = cuda(wl.rmsnorm_inputs(96, 1024, "bf16", seed=710))
    grads = []
    for save in (False, True):
        x = d["x"].clone().requires_grad_(True)
        w = d["w"].clone().requires_grad_(True)
        y = fq.rmsnorm(x, w, save_rstd=save)
        (y.float() * d["g"].float()).sum().backward()
        grads.append((y.detach(), x.grad, w.grad))
    assert torch.equal(grads[0][0], grads[1][0])
    assert_storage_close(grads[1][1], grads[0][1].cpu(), "dx")
    assert_storage_close(grads[1][2], grads[0][2].cpu(), "dw")


# LayerNorm: shapes that reach the register-resident, the TMA-fed and the scalar kernels
LN_CASES = [
    # M, N, dtype, bias, misalign
    (300, 256, "bf16", True, False),
    (129, 2048, "fp16", True, False),
    (4097, 4096, "bf16", True, False),   # TMA-fed wide rows
    (4100, 1024, "fp16", False, False),  # TMA-fed, no bias
    (4099, 3000, "bf16", True, False),   # TMA-fed, two warps per row, ragged last vectors
    (4097, 2056, "fp16", False, False),  # two warps per row, the second holding one vector
    (4096, 1536, "bf16", True, False),   # TMA-fed, one warp per row, partly filled slots
    (4096, 512, "bf16", True, False),    # many narrow rows: register-resident kernel
    (77, 100, "bf16", True, False),      # odd width: scalar
    (9, 5000, "bf16", True, False),      # wider than the register kernel: scalar
    (60, 512, "fp16", True, True),       # misaligned: scalar
]


@pytest.mark.parametrize("case", LN_CASES, ids=lambda c: "M%d-N%d-%s-b%d-mis%d" % c)
def test_layernorm_parity(orc, cuda_ok, case):
    M, N, dt, bias, mis = case
    d = wl.rmsnorm_inputs(M, N, dt, seed=800 + M)
    b = (d["w"].float() - 1.0).to(d["w"].dtype) if bias else None
    y_ref, _, _ = orc.layernorm_fwd(d["x"], d["w"], b)
    g = cuda(d)
    x = misalign(g["x"]) if mis else g["x"]
    y = fq.layernorm_fwd(x, g["w"], None if b is None else b.cuda())
    torch.cuda.synchronize()
    assert_storage_close(y, y_ref)
    assert fq.device_status(clear=True) == 0


def test_rmsnorm_bwd_deterministic(cuda_ok):
    d = cuda(wl.rmsnorm_inputs(1000, 4096, "bf16", seed=550))
    a = fq.rmsnorm_bwd(d["x"], d["w"], d["g"])
    b = fq.rmsnorm_bwd(d["x"], d["w"], d["g"])
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_rmsnorm_bwd_empty_gives_zero_dw(cuda_ok):
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(256, dtype=torch.bfloat16, device="cuda")
    dx, dw, dw32 = fq.rmsnorm_bwd(x, w, x)
    assert dx.shape == (0, 256) and torch.equal(dw32.cpu(), torch.zeros(256))


def test_autograd_wrapper(orc, cuda_ok):
    d = wl.rmsnorm_inputs(48, 256, "bf16", seed=560)
    x = d["x"].cuda().requires_grad_(True)
    w = d["w"].cuda().requires_grad_(True)
    y = fq.rmsnorm(x, w)
    y.backward(d["g"].cuda())
    dx_ref, dw_ref, _ = orc.rmsnorm_bwd(d["x"], d["w"], d["g"])
    assert_storage_close(y.detach(), orc.rmsnorm_fwd(d["x"], d["w"]))
    assert_storage_close(x.grad, dx_ref, "dx")
    assert_within_one_ulp(w.grad, dw_ref)


def test_device_status_clean_after_runs(cuda_ok):
    assert fq.device_status(clear=True) == 0


# ----------------------------------------------------------------------------------- TMA prologue kernel
TMA_CASES = [
    # T, Hq, Hk, dtype, table, stride_extra
    (4096, 32, 8, "bf16", "fp32", 0),     # the measured workload
    (1, 1, 0, "bf16", "fp32", 0),         # a single row
    (3, 1, 0, "fp16", "fp32", 0),         # H = 1: every row of a stage is a different token
    (97, 1, 1, "bf16", "bf16", 0),        # H = 2, 16-bit tables
    (50, 64, 8, "bf16", "fp32", 0),       # large H, stages span token boundaries
    (211, 5, 3, "fp16", "fp16", 0),       # rows not a multiple of the 64-row stage
    (65, 3, 1, "bf16", "fp32", 2 * 128),  # q/k slice of a wider row: one copy per token segment
    (300, 6, 2, "bf16", "fp32", 8),       # odd token stride (still 16-byte aligned)
]


@pytest.mark.parametrize("kernel", ["tma", "generic"])
@pytest.mark.parametrize("case", TMA_CASES, ids=lambda c: "T%d-%d+%d-%s-%s-x%d" % c)
def test_prologue_tma_kernel_parity(orc, cuda_ok, monkeypatch, case, kernel):
    T, Hq, Hk, dt, tdt, extra = case
    if kernel == "generic":
        monkeypatch.setenv("FQ_PROLOGUE_KERNEL", "generic")
    else:
        monkeypatch.delenv("FQ_PROLOGUE_KERNEL", raising=False)
    H = Hq + Hk
    ts = None if extra == 0 else H * 128 + extra
    d = wl.qk_inputs(T, Hq, Hk, 128, dt, tdt, seed=700 + T, std=2.0, token_stride=ts)
    q_ref, s_ref = orc.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], Hq, Hk)
    g = cuda(d)
    q, s = fq.qk_norm_rope_quant(g["qk"], g["wq"], g["wk"], g["cos"], g["sin"], Hq, Hk)
    torch.cuda.synchronize()
    assert_scale_close(s, s_ref)
    assert_codes_close(q, q_ref)
    assert fq.device_status(clear=True) == 0


@pytest.mark.parametrize("case", [(4096, 32, 8), (1000, 3, 1), (333, 64, 8), (5, 1, 0)],
                         ids=lambda c: "T%d-%d+%d" % c)
def test_prologue_tma_writes_every_row(orc, cuda_ok, monkeypatch, case):
    """Every chunk of rows is processed exactly once, whichever CTA takes it over: outputs pre-filled
    with NaN codes and NaN scales hold no leftover after the call, twice in a row on the same buffers
    with different inputs (so a skipped chunk cannot pass on the previous call's values)."""
    T, Hq, Hk = case
    monkeypatch.delenv("FQ_PROLOGUE_KERNEL", raising=False)
    H = Hq + Hk
    q = torch.full((T, H, 128), 0x7F, dtype=torch.uint8, device="cuda")
    s = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    for seed in (901, 902):
        d = wl.qk_inputs(T, Hq, Hk, 128, "bf16", "fp32", seed=seed + T, std=2.0)
        q_ref, s_ref = orc.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], Hq, Hk)
        g = cuda(d)
        fq.qk_norm_rope_quant(g["qk"], g["wq"], g["wk"], g["cos"], g["sin"], Hq, Hk, q_out=q, scale=s)
        torch.cuda.synchronize()
        assert not bool(torch.isnan(s).any())
        assert_scale_close(s, s_ref)
        assert_codes_close(q, q_ref)
    assert fq.device_status(clear=True) == 0


@pytest.mark.parametrize("rpb", [1, 8, 40, 128])
@pytest.mark.parametrize("case", [(37, 32, 8, "bf16", "fp32"), (21, 6, 2, "fp16", "fp16"), (9, 3, 0, "bf16", "bf16")],
                         ids=lambda c: "T%d-%d+%d-%s-%s" % c)
def test_prologue_design_blocks(orc, cuda_ok, monkeypatch, case, rpb):
    """The Ch.28 page's designs (one CTA per block of 1, 8, a token's 40, or 128 rows; ragged last
    blocks): against the oracle, and bit for bit the generic prologue kernel (same arithmetic)."""
    T, Hq, Hk, dt, tdt = case
    d = wl.qk_inputs(T, Hq, Hk, 128, dt, tdt, seed=820 + T, std=2.0)
    q_ref, s_ref = orc.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], Hq, Hk)
    g = cuda(d)
    q, s = fq.qk_norm_rope_quant_blocks(g["qk"], g["wq"], g["wk"], g["cos"], g["sin"], Hq, Hk, rpb)
    torch.cuda.synchronize()
    assert_scale_close(s, s_ref)
    assert_codes_close(q, q_ref)
    monkeypatch.setenv("FQ_PROLOGUE_KERNEL", "generic")
    q2, s2 = fq.qk_norm_rope_quant(g["qk"], g["wq"], g["wk"], g["cos"], g["sin"], Hq, Hk)
    assert torch.equal(q, q2) and torch.equal(s, s2)


def test_prologue_tma_matches_generic_kernel(cuda_ok, monkeypatch):
    """Both kernels on identical inputs: scales within 1e-6 relative, codes at most one step apart."""
    d = cuda(wl.qk_inputs(777, 32, 8, 128, "bf16", "fp32", seed=790, std=2.0))
    monkeypatch.delenv("FQ_PROLOGUE_KERNEL", raising=False)
    q1, s1 = fq.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], 32, 8)
    monkeypatch.setenv("FQ_PROLOGUE_KERNEL", "generic")
    q2, s2 = fq.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], 32, 8)
    assert_scale_close(s1, s2.cpu(), rel=1e-6)
    assert_codes_close(q1, q2.cpu())


# ----------------------------------------------------------------------------------- failure detection
def test_strict_mode_reports_a_bounded_wait_failure(orc, cuda_ok):
    """In strict mode a compute call waits for its stream and returns FQ_ERR_DEVICE when a bounded
    wait gave up since the status word was last read (here: the diagnostic wait, which nothing can
    complete); the word is cleared by that report and the next call succeeds with correct results."""
    import ctypes

    from fp8_quant_memory_gb300 import _capi

    d = wl.qk_inputs(64, 8, 2, 128, seed=881)
    g = cuda(d)
    q_ref, s_ref = orc.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], 8, 2)
    assert fq.device_status(clear=True) == 0
    prev = fq.set_strict(True)
    try:
        _capi.call("fq_check_bounded_wait", ctypes.c_uint(50), fq._stream(g["qk"].device))
        with pytest.raises(_capi.FqError) as err:
            fq.qk_norm_rope_quant(g["qk"], g["wq"], g["wk"], g["cos"], g["sin"], 8, 2)
        assert err.value.status == _capi.FQ_ERR_DEVICE
        q, s = fq.qk_norm_rope_quant(g["qk"], g["wq"], g["wk"], g["cos"], g["sin"], 8, 2)
        assert_scale_close(s, s_ref)
        assert_codes_close(q, q_ref)
    finally:
        fq.set_strict(prev)
    assert fq.device_status(clear=True) == 0


def test_bounded_wait_gives_up_and_context_stays_usable(orc, cuda_ok):
    """A wait that nothing completes ends after its limit and reports through the status word; the
    next calls on the same context run and are correct."""
    import time

    t0 = time.perf_counter()
    word = fq.check_bounded_wait(50)
    elapsed = time.perf_counter() - t0
    assert word & 1
    assert 0.04 <= elapsed < 5.0
    assert fq.device_status(clear=True) == 0
    d = wl.qk_inputs(64, 8, 2, 128, seed=880)
    q_ref, s_ref = orc.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], 8, 2)
    g = cuda(d)
    q, s = fq.qk_norm_rope_quant(g["qk"], g["wq"], g["wk"], g["cos"], g["sin"], 8, 2)
    assert_scale_close(s, s_ref)
    assert_codes_close(q, q_ref)
    assert fq.device_status(clear=True) == 0


# ----------------------------------------------------------------------------------- TMA row-stream kernels
def _rows_kernel(monkeypatch, kernel):
    if kernel in ("generic", "staged"):
        monkeypatch.setenv("FQ_ROWS_KERNEL", kernel)
    else:
        monkeypatch.delenv("FQ_ROWS_KERNEL", raising=False)


@pytest.mark.parametrize("kernel", ["tma", "staged", "generic"])
@pytest.mark.parametrize("case", [(4099, 256, "bf16"), (4500, 1024, "bf16"), (4097, 4096, "fp16"), (5000, 64, "fp16"),
                                  (4608, 2048, "bf16"), (4103, 8192, "bf16"), (4096, 1032, "fp16"),
                                  (4097, 3000, "bf16"), (4098, 2056, "fp16")],
                         ids=lambda c: "M%d-N%d-%s" % c)
def test_rmsnorm_fwd_stream_kernel(orc, cuda_ok, monkeypatch, case, kernel):
    _rows_kernel(monkeypatch, kernel)
    M, N, dt = case
    d = wl.rmsnorm_inputs(M, N, dt, seed=900 + M)
    g = cuda(d)
    y = fq.rmsnorm_fwd(g["x"], g["w"])
    assert_storage_close(y, orc.rmsnorm_fwd(d["x"], d["w"]))
    assert fq.device_status(clear=True) == 0


@pytest.mark.parametrize("case", [(5000, 192, 64, "fp16", "fp16", 32), (4097, 128, 128, "bf16", "fp32", 1),
                                  (4200, 512, 64, "bf16", "bf16", 8), (4100, 256, 32, "fp16", "fp32", 4),
                                  (4099, 1024, 128, "bf16", "bf16", 1), (4096, 96, 0, "bf16", "bf16", 1),
                                  (4101, 2048, 64, "bf16", "fp32", 2)],
                         ids=lambda c: "M%d-N%d-R%d-%s-%s-h%d" % c)
@pytest.mark.parametrize("kernel", ["tma", "generic"])
def test_rmsnorm_rope_stream_kernel(orc, cuda_ok, monkeypatch, case, kernel):
    _rows_kernel(monkeypatch, kernel)
    M, N, R, dt, tdt, hpt = case
    d = wl.rows_inputs(M, N, R, dt, tdt, seed=950 + M, heads_per_token=hpt)
    g = cuda(d)
    y = fq.rmsnorm_rope(g["x"], g["w"], g["cos"], g["sin"])
    assert_rope_close(y, orc.rmsnorm_rope(d["x"], d["w"], d["cos"], d["sin"]),
                      orc.rmsnorm_fwd(d["x"], d["w"]), d["cos"], d["sin"])
    assert fq.device_status(clear=True) == 0


# ----------------------------------------------------------------------------------- streaming floor
@pytest.mark.parametrize("n16", [1, 511, 513, 5000, 163840 * 16])
def test_stream_floor_output(cuda_ok, n16):
    """The size-matched copy the benchmark times beside the prologue does exactly its stated work:
    every input vector read once, out word k = in word k XOR in word k + 2 (ragged last chunk too)."""
    g = torch.Generator().manual_seed(n16)
    x = torch.randint(-2 ** 31, 2 ** 31 - 1, (n16, 4), dtype=torch.int32, generator=g)
    out = fq.stream_floor(x.cuda())
    torch.cuda.synchronize()
    expect = torch.stack([x[:, 0] ^ x[:, 2], x[:, 1] ^ x[:, 3]], 1)
    assert torch.equal(out.cpu().view(torch.int32).view(n16, 2), expect)
    assert fq.device_status(clear=True) == 0
