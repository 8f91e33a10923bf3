"""Guard bands around every output of every libfq entry point (tests/guards.py): ragged last stages
(1, 3, 211, 4097 tokens; row counts one past a stage), token strides wider than the heads, rows past
the end of the tensor that the bulk copies zero-fill or skip, and workspaces passed at exactly the
size the library asks for. Each guarded call must leave the bands untouched and give the same bytes
as the same call on ordinary tensors; the prologue cases are also compared with the oracle.
"""
import pytest
import torch

import fp8_quant_memory_gb300 as fq
from fp8_quant_memory_gb300 import _capi
from fp8_quant_memory_gb300 import workloads as wl
from guards import Guarded, check_all
from parity import assert_codes_close, assert_scale_close

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def cuda(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def same(a, b, what):
    assert torch.equal(a.view(torch.uint8) if a.dtype != torch.uint8 else a,
                       b.view(torch.uint8) if b.dtype != torch.uint8 else b), f"{what}: guarded call differs"


# ----------------------------------------------------------------------------------------- prologue
PROLOGUE = [
    # T, Hq, Hk, dtype, table, extra token stride, kernel
    (1, 32, 8, "bf16", "fp32", 0, "tma"),
    (3, 32, 8, "bf16", "fp32", 0, "tma"),
    (211, 5, 3, "fp16", "fp16", 0, "tma"),
    (4097, 32, 8, "bf16", "fp32", 0, "tma"),
    (4097, 32, 8, "bf16", "fp32", 0, "generic"),
    (5, 1, 0, "bf16", "fp32", 0, "tma"),          # H = 1: every row its own token
    (97, 1, 1, "bf16", "bf16", 0, "tma"),
    (333, 64, 8, "bf16", "fp32", 0, "tma"),
    (65, 3, 1, "bf16", "fp32", 2 * 128, "tma"),   # q/k slice of a wider row (generic kernel)
    (300, 6, 2, "bf16", "fp32", 8, "tma"),
]


@pytest.mark.parametrize("case", PROLOGUE, ids=lambda c: "T%d-%d+%d-%s-%s-x%d-%s" % c)
def test_prologue_outputs_stay_inside(orc, cuda_ok, monkeypatch, case):
    T, Hq, Hk, dt, tdt, extra, kernel = case
    if kernel == "generic":
        monkeypatch.setenv("FQ_PROLOGUE_KERNEL", "generic")
    else:
        monkeypatch.delenv("FQ_PROLOGUE_KERNEL", raising=False)
    H = Hq + Hk
    ts = None if extra == 0 else H * 128 + extra
    d = wl.qk_inputs(T, Hq, Hk, 128, dt, tdt, seed=1300 + T, std=2.0, token_stride=ts)
    q_ref, s_ref = orc.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], Hq, Hk)
    g = cuda(d)
    q = Guarded((T, H, 128), torch.uint8, fill=0x7F)
    s = Guarded((T, H), torch.float32, fill=float("nan"))
    fq.qk_norm_rope_quant(g["qk"], g["wq"], g["wk"], g["cos"], g["sin"], Hq, Hk, q_out=q.t, scale=s.t)
    check_all(q=q, scale=s)
    assert_scale_close(s.t, s_ref)
    assert_codes_close(q.t, q_ref)
    assert fq.device_status(clear=True) == 0


@pytest.mark.parametrize("rpb", [1, 8, 40, 128])
def test_prologue_blocks_outputs_stay_inside(orc, cuda_ok, rpb):
    T, Hq, Hk = 37, 32, 8
    d = wl.qk_inputs(T, Hq, Hk, 128, "bf16", "fp32", seed=1400, std=2.0)
    q_ref, s_ref = orc.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], Hq, Hk)
    g = cuda(d)
    q = Guarded((T, Hq + Hk, 128), torch.uint8)
    s = Guarded((T, Hq + Hk), torch.float32)
    fq.qk_norm_rope_quant_blocks(g["qk"], g["wq"], g["wk"], g["cos"], g["sin"], Hq, Hk, rpb, q_out=q.t, scale=s.t)
    check_all(q=q, scale=s)
    assert_scale_close(s.t, s_ref)
    assert_codes_close(q.t, q_ref)


# ----------------------------------------------------------------------------------------- row calls
FWD = [(1, 4096, "bf16"), (4097, 1024, "bf16"), (4100, 8192, "bf16"), (4099, 192, "fp16"), (37, 100, "bf16"),
       (45, 2048, "fp16"), (4097, 4096, "bf16")]


@pytest.mark.parametrize("case", FWD, ids=lambda c: "M%d-N%d-%s" % c)
def test_rmsnorm_fwd_outputs_stay_inside(cuda_ok, case):
    M, N, dt = case
    d = cuda(wl.rmsnorm_inputs(M, N, dt, seed=1500 + M))
    y = Guarded((M, N), DT[dt])
    fq.rmsnorm_fwd(d["x"], d["w"], out=y.t)
    y2 = Guarded((M, N), DT[dt])
    r2 = Guarded((M,), torch.float32)
    fq.rmsnorm_fwd_rstd(d["x"], d["w"], out=y2.t, rstd=r2.t)
    check_all(y=y, y_rstd=y2, rstd=r2)
    same(y.t, fq.rmsnorm_fwd(d["x"], d["w"]), "rmsnorm_fwd")
    yy, rr = fq.rmsnorm_fwd_rstd(d["x"], d["w"])
    same(y2.t, yy, "rmsnorm_fwd_rstd y")
    same(r2.t, rr, "rmsnorm_fwd_rstd rstd")
    assert fq.device_status(clear=True) == 0


ROPE = [(4097, 192, 64, "fp16", "fp16"), (4100, 1024, 128, "bf16", "bf16"), (33, 100, 20, "bf16", "bf16"),
        (64, 512, 64, "bf16", "fp32"), (4096 + 33, 1536, 256, "bf16", "fp32")]


@pytest.mark.parametrize("case", ROPE, ids=lambda c: "M%d-N%d-R%d-%s-%s" % c)
def test_rmsnorm_rope_outputs_stay_inside(cuda_ok, case):
    M, N, R, dt, tdt = case
    d = cuda(wl.rows_inputs(M, N, R, dt, tdt, seed=1600 + M))
    y = Guarded((M, N), DT[dt])
    fq.rmsnorm_rope(d["x"], d["w"], d["cos"], d["sin"], out=y.t)
    check_all(y=y)
    same(y.t, fq.rmsnorm_rope(d["x"], d["w"], d["cos"], d["sin"]), "rmsnorm_rope")
    assert fq.device_status(clear=True) == 0


QUANT = [  # M, N, R, dtype, table, group size (None: one scale per row)
    (4097, 4096, 128, "bf16", "bf16", None), (4096 + 5, 1024, 64, "bf16", "fp32", None),
    (256, 512, 64, "bf16", "bf16", None), (33, 100, 20, "bf16", "bf16", None),
    (4100, 1536, 256, "bf16", "bf16", None), (4097, 4096, 128, "bf16", "bf16", 128),
    (4100, 2048, 64, "fp16", "fp16", 512), (256, 512, 64, "bf16", "bf16", 128), (33, 96, 16, "bf16", "bf16", 32),
]


@pytest.mark.parametrize("want_y", [True, False])
@pytest.mark.parametrize("case", QUANT, ids=lambda c: "M%d-N%d-R%d-%s-%s-g%s" % c)
def test_rmsnorm_rope_quant_outputs_stay_inside(cuda_ok, case, want_y):
    M, N, R, dt, tdt, gs = case
    d = cuda(wl.rows_inputs(M, N, R, dt, tdt, seed=1700 + M))
    y = Guarded((M, N), DT[dt]) if want_y else None
    q = Guarded((M, N), torch.uint8)
    s = Guarded((M,) if gs is None else (M, N // gs), torch.float32)
    if gs is None:
        fq.rmsnorm_rope_quant(d["x"], d["w"], d["cos"], d["sin"], want_y=want_y, y=None if y is None else y.t,
                              q=q.t, scale=s.t)
        y2, q2, s2 = fq.rmsnorm_rope_quant(d["x"], d["w"], d["cos"], d["sin"], want_y=want_y)
    else:
        fq.rmsnorm_rope_quant_groups(d["x"], d["w"], d["cos"], d["sin"], gs, want_y=want_y,
                                     y=None if y is None else y.t, q=q.t, scale=s.t)
        y2, q2, s2 = fq.rmsnorm_rope_quant_groups(d["x"], d["w"], d["cos"], d["sin"], gs, want_y=want_y)
    check_all(y=y, q=q, scale=s)
    same(q.t, q2, "codes")
    same(s.t, s2, "scales")
    if want_y:
        same(y.t, y2, "y")
    assert fq.device_status(clear=True) == 0


LN = [(4097, 4096, "bf16", True), (4100, 1024, "fp16", False), (37, 100, "bf16", True), (64, 2048, "bf16", True)]


@pytest.mark.parametrize("case", LN, ids=lambda c: "M%d-N%d-%s-bias%d" % c)
def test_layernorm_outputs_stay_inside(cuda_ok, case):
    M, N, dt, bias = case
    h = wl.rmsnorm_inputs(M, N, dt, seed=1800 + M)
    d = cuda({"x": h["x"], "g": h["w"], "b": (h["w"].float() - 1.0).to(DT[dt])})
    b = d["b"] if bias else None
    y = Guarded((M, N), DT[dt])
    fq.layernorm_fwd(d["x"], d["g"], b, out=y.t)
    check_all(y=y)
    same(y.t, fq.layernorm_fwd(d["x"], d["g"], b), "layernorm_fwd")
    assert fq.device_status(clear=True) == 0


# ----------------------------------------------------------------------------------------- backward
BWD = [(1, 4096, "bf16"), (4097, 4096, "bf16"), (333, 1032, "fp16"), (37, 100, "bf16"), (513, 8192, "bf16"),
       (300, 2048, "bf16")]


def _bwd_guarded(d, M, N, dt, rstd=None, noalloc=False):
    dx = Guarded((M, N), DT[dt])
    dw = Guarded((N,), DT[dt])
    dw32 = Guarded((N,), torch.float32)
    x, w, g = d["x"], d["w"], d["g"]
    code = fq._dtype("guards", x)
    stream = fq._stream(x.device)
    P = fq._ptr
    ws = None
    if noalloc:
        _capi.call("fq_rmsnorm_bwd_noalloc", P(x), P(w), P(g), P(dx.t), P(dw.t), P(dw32.t), M, N, code, 1e-6, stream)
    else:
        need = fq.rmsnorm_bwd_workspace_bytes(M, N)
        ws = Guarded((need,), torch.uint8)
        if rstd is None:
            _capi.call("fq_rmsnorm_bwd", P(x), P(w), P(g), P(dx.t), P(dw.t), P(dw32.t), P(ws.t), need, M, N, code,
                       1e-6, stream)
        else:
            _capi.call("fq_rmsnorm_bwd_rstd", P(x), P(w), P(g), P(rstd), P(dx.t), P(dw.t), P(dw32.t), P(ws.t), need,
                       M, N, code, stream)
    check_all(dx=dx, dw=dw, dw_f32=dw32, workspace=ws)
    return dx.t, dw.t, dw32.t


@pytest.mark.parametrize("case", BWD, ids=lambda c: "M%d-N%d-%s" % c)
def test_rmsnorm_bwd_outputs_stay_inside(cuda_ok, case):
    M, N, dt = case
    d = cuda(wl.rmsnorm_inputs(M, N, dt, seed=1900 + M))
    dx, dw, dw32 = _bwd_guarded(d, M, N, dt)
    ex, ew, e32 = fq.rmsnorm_bwd(d["x"], d["w"], d["g"])
    same(dx, ex, "dx")
    same(dw, ew, "dw")
    same(dw32, e32, "dw_f32")
    rstd = fq.rmsnorm_fwd_rstd(d["x"], d["w"])[1]
    dx, dw, dw32 = _bwd_guarded(d, M, N, dt, rstd=rstd)
    ex, ew, e32 = fq.rmsnorm_bwd_rstd(d["x"], d["w"], d["g"], rstd)
    same(dx, ex, "dx (saved rstd)")
    same(dw32, e32, "dw_f32 (saved rstd)")
    assert fq.device_status(clear=True) == 0


@pytest.mark.parametrize("case", [(4097, 4096, "bf16"), (37, 100, "bf16")], ids=lambda c: "M%d-N%d-%s" % c)
def test_rmsnorm_bwd_noalloc_outputs_stay_inside(cuda_ok, case):
    M, N, dt = case
    d = cuda(wl.rmsnorm_inputs(M, N, dt, seed=2000 + M))
    dx, dw, dw32 = _bwd_guarded(d, M, N, dt, noalloc=True)
    ex, ew, e32 = fq.rmsnorm_bwd(d["x"], d["w"], d["g"])
    same(dx, ex, "dx")
    same(dw32, e32, "dw_f32")
    assert fq.device_status(clear=True) == 0


@pytest.mark.parametrize("n16", [1, 511, 513, 12345])
def test_stream_floor_output_stays_inside(cuda_ok, n16):
    inp = torch.randint(0, 256, (n16 * 16,), dtype=torch.uint8, device="cuda")
    out = Guarded((n16 * 8,), torch.uint8)
    fq.stream_floor(inp, out=out.t)
    check_all(out=out)
    same(out.t, fq.stream_floor(inp), "stream_floor")
